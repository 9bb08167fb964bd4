// Sequence-wise balance statistics of a routing step (DeepSeek-V3 Technical
// Report, learn.ifs.name summary, bias paragraph: beside the per-expert bias a
// tiny sequence-wise balancing loss remains, against extreme imbalance inside
// one sequence). For a sequence of T_s consecutive tokens and expert i:
//   loads_i = pairs (t, k) of the sequence routed to i
//   P_i     = (1/T_s) sum_t s_{i,t} / sum_j s_{j,t}   (affinities over all N)
//   stat    = sum_i f_i P_i,  f_i = N loads_i / (K T_s)
// The loss weight is the caller's. Every sum runs in a fixed order, so the
// results are reproducible bit for bit:
//   partial   one block per chunk of up to 64 tokens of one sequence: row sums
//             (warp per token, fixed shuffle tree), then a thread per expert
//             sums s / rowsum over the chunk's tokens in token order; the
//             chunk's loads come from shared-memory integer counters;
//   final     one block per sequence: the chunks' partial sums in chunk order,
//             then sum_i f_i P_i by a fixed tree over the block.
// HBM bound: the scores are read once (T * N * 4 bytes).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kBalChunk = 64;   // tokens per partial block

__global__ void __launch_bounds__(256) balance_partial_kernel(const float* __restrict__ scores,
                                                              const int32_t* __restrict__ idx, int64_t T, int N,
                                                              int K, int64_t seq_len, int64_t chunks_per_seq,
                                                              float* __restrict__ part_p, int32_t* __restrict__ part_c) {
    extern __shared__ int bal_sm[];
    int* cnt = bal_sm;                                          // [N]
    float* rowsum = reinterpret_cast<float*>(bal_sm + N);      // [kBalChunk]
    const int64_t c = blockIdx.x;
    const int64_t s = c / chunks_per_seq, j = c - s * chunks_per_seq;
    const int64_t seq_end = min(T, (s + 1) * seq_len);
    const int64_t t0 = s * seq_len + j * kBalChunk;
    const int64_t t1 = min(seq_end, t0 + kBalChunk);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < N; i += blockDim.x) cnt[i] = 0;
    // row sums: warp per token, lanes over experts, then a fixed xor tree
    for (int64_t t = t0 + w; t < t1; t += blockDim.x >> 5) {
        float acc = 0.0f;
        for (int i = lane; i < N; i += 32) acc += __ldg(scores + t * N + i);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) rowsum[t - t0] = acc;
    }
    __syncthreads();
    for (int64_t p = t0 * K + threadIdx.x; p < t1 * K; p += blockDim.x) {
        const int e = __ldg(idx + p);
        if (e >= 0 && e < N) atomicAdd(&cnt[e], 1);
        else report(MOE_ERR_DEVICE_DATA);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        float acc = 0.0f;
        for (int64_t t = t0; t < t1; ++t) acc += __fdiv_rn(__ldg(scores + t * N + i), rowsum[t - t0]);
        part_p[c * N + i] = acc;
        part_c[c * N + i] = cnt[i];
    }
}

__global__ void __launch_bounds__(256) balance_final_kernel(const float* __restrict__ part_p,
                                                            const int32_t* __restrict__ part_c, int64_t T, int N,
                                                            int K, int64_t seq_len, int64_t chunks_per_seq,
                                                            int32_t* __restrict__ seq_loads,
                                                            float* __restrict__ seq_prob, float* __restrict__ seq_stat) {
    __shared__ float red[256];
    const int64_t s = blockIdx.x;
    const int64_t t0 = s * seq_len, t1 = min(T, t0 + seq_len);
    const int64_t n_chunks = (t1 - t0 + kBalChunk - 1) / kBalChunk;
    const int64_t c0 = s * chunks_per_seq;
    const float Ts = float(t1 - t0);
    float mine = 0.0f;
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        float p = 0.0f;
        int32_t n = 0;
        for (int64_t c = c0; c < c0 + n_chunks; ++c) {
            p += part_p[c * N + i];
            n += part_c[c * N + i];
        }
        const float P = __fdiv_rn(p, Ts);
        const float f = __fdiv_rn(float(N) * float(n), float(K) * Ts);
        seq_loads[s * N + i] = n;
        seq_prob[s * N + i] = P;
        mine = __fmaf_rn(f, P, mine);
    }
    red[threadIdx.x] = mine;
    __syncthreads();
    for (int o = blockDim.x >> 1; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) seq_stat[s] = red[0];
}

}  // namespace

size_t balance_ws_bytes(int64_t T, int N, int64_t seq_len) {
    if (T <= 0 || seq_len <= 0) return 256;
    const int64_t S = (T + seq_len - 1) / seq_len;
    const int64_t cps = (seq_len + kBalChunk - 1) / kBalChunk;
    const size_t chunks = size_t(S) * size_t(cps);
    return (chunks * size_t(N) * 8 + 255) / 256 * 256;
}

cudaError_t launch_balance(const float* scores, const int32_t* topk_idx, int64_t T, int N, int K, int64_t seq_len,
                           int32_t* seq_loads, float* seq_prob, float* seq_stat, void* ws, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int64_t S = (T + seq_len - 1) / seq_len;
    const int64_t cps = (seq_len + kBalChunk - 1) / kBalChunk;
    const int64_t last_chunks = (T - (S - 1) * seq_len + kBalChunk - 1) / kBalChunk;
    const int64_t chunks = (S - 1) * cps + last_chunks;
    float* part_p = reinterpret_cast<float*>(ws);
    int32_t* part_c = reinterpret_cast<int32_t*>(part_p + size_t(S) * size_t(cps) * size_t(N));
    const size_t smem = size_t(N) * 4 + kBalChunk * 4;
    balance_partial_kernel<<<unsigned(chunks), 256, smem, stream>>>(scores, topk_idx, T, N, K, seq_len, cps, part_p,
                                                                   part_c);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    balance_final_kernel<<<unsigned(S), 256, 0, stream>>>(part_p, part_c, T, N, K, seq_len, cps, seq_loads, seq_prob,
                                                          seq_stat);
    return cudaGetLastError();
}

}  // namespace moe
