// Routing (DeepSeek-V3 Technical Report: learn.ifs.name summary, MoE and bias
// paragraphs; nlp-lineage.vercel.app, "The notation"):
//   z_{t,i} = u_t . e_i                 tensor cores (tcgen05), fp32 accumulation
//   s_{t,i} = 1 / (1 + exp(-z))         affinity
//   key     = s + b_i                   the bias only steers the choice
//   chosen  = top-K keys (ties: lower index), optionally only inside the
//             topk_groups groups with the largest sum of their two best keys
//   g       = s / sum_chosen s          gates from the raw affinities
//   loads_i = number of tokens choosing i
//
// fp32 centroids are split exactly into three bf16 terms (hi + mid + lo = e,
// each product with a bf16 token value exact in fp32), so the gate runs as a
// bf16 GEMM over K = 3d with fp32 accumulation; bf16 centroids need one term.
// The split operand keeps the three terms of each 64-column block side by side
// (hi, mid, lo), so a tile of u is fetched once and feeds three consecutive K
// steps.
// The GEMM is split along K over enough blocks to fill the GPU; a warp per
// token then sums the partial logits in a fixed order and selects.
#include <cuda_bf16.h>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

__global__ void split_centroids_kernel(const void* __restrict__ cent, int f32, int N, int n_pad, int d, int terms,
                                       uint16_t* __restrict__ out) {
    const int64_t total = int64_t(n_pad) * d;
    const int64_t ld = int64_t(terms) * d;
    for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; p < total; p += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = p / d, j = p - i * d;
        uint16_t* row = out + i * ld;
        if (i >= N) {
            for (int t = 0; t < terms; ++t) row[t * d + j] = 0;
            continue;
        }
        if (!f32) {
            row[j] = reinterpret_cast<const uint16_t*>(cent)[p];
            continue;
        }
        const float x = reinterpret_cast<const float*>(cent)[p];
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const float r1 = x - __bfloat162float(hi);          // exact
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);        // exact, fits 8 bits
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        uint16_t* blk = row + int64_t(j / 64) * 3 * 64 + (j % 64);
        blk[0] = __bfloat16_as_ushort(hi);
        blk[64] = __bfloat16_as_ushort(mid);
        blk[128] = __bfloat16_as_ushort(lo);
    }
}

// Lane-local then warp-wide arg-max with ties to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

// One warp per token. Lane l holds experts i = 32j + l, j < J.
template <int J>
__global__ void __launch_bounds__(256) route_select_kernel(const float* __restrict__ zpart, int splits, int64_t T,
                                                           int n_pad, const float* __restrict__ bias, int N, int K,
                                                           int n_groups, int topk_groups, int32_t* __restrict__ topk_idx,
                                                           float* __restrict__ gates, int32_t* __restrict__ loads,
                                                           float* __restrict__ scores,
                                                           float* __restrict__ logits) {
    extern __shared__ int sm[];
    int* hist = sm;                                            // [N]
    float* keys_sm = reinterpret_cast<float*>(sm + N);         // [8][N] when grouped
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < N; i += blockDim.x) hist[i] = 0;
    __syncthreads();

    float b[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int i = 32 * j + lane;
        b[j] = i < N ? __ldg(bias + i) : 0.0f;
    }
    const int per_group = N / n_groups;
    const int64_t plane = T * int64_t(n_pad);

    for (int64_t t = int64_t(blockIdx.x) * 8 + w; t < T; t += int64_t(gridDim.x) * 8) {
        float s[J], key[J];
        // bit j: expert 32j + lane is out of the running (past N, outside the kept
        // groups, or already chosen)
        uint32_t excl = 0;
        // z of each of the lane's experts: the split-K partials added in split order;
        // a split's J loads are issued together (small batches take many splits)
        float zj[J];
        const float* zt = zpart + t * n_pad + lane;
#pragma unroll
        for (int j = 0; j < J; ++j) zj[j] = 32 * j + lane < N ? __ldg(zt + 32 * j) : 0.0f;
        for (int p = 1; p < splits; ++p) {
            float v[J];
#pragma unroll
            for (int j = 0; j < J; ++j) v[j] = 32 * j + lane < N ? __ldg(zt + p * plane + 32 * j) : 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j) zj[j] += v[j];
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int i = 32 * j + lane;
            const float z = zj[j];
            if (i >= N) excl |= 1u << j;
            s[j] = __fdiv_rn(1.0f, 1.0f + expf(-z));
            const float kv = s[j] + b[j];
            // a NaN key (NaN token or bias) ranks below every number: it can still be
            // chosen, last, so every token keeps exactly K valid experts
            key[j] = (i < N && kv == kv) ? kv : -INFINITY;
            if (scores && i < N) scores[t * N + i] = s[j];
            if (logits && i < N) logits[t * N + i] = z;
        }
        if (n_groups > 1) {
            float* ks = keys_sm + w * N;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int i = 32 * j + lane;
                if (i < N) ks[i] = key[j];
            }
            __syncwarp();
            float gscore = -INFINITY;
            if (lane < n_groups) {
                float t1 = -INFINITY, t2 = -INFINITY;
                for (int p = 0; p < per_group; ++p) {
                    const float v = ks[lane * per_group + p];
                    if (v > t1) {
                        t2 = t1;
                        t1 = v;
                    } else if (v > t2) {
                        t2 = v;
                    }
                }
                gscore = t1 + t2;
                if (!(gscore == gscore)) gscore = -INFINITY;   // +inf + -inf
            }
            __syncwarp();
            // topk_groups rounds over the groups not kept yet; a lane past n_groups or
            // holding a kept group offers no candidate, so every round keeps a new group
            uint32_t keep = 0;
            bool kept_me = false;
            for (int r = 0; r < topk_groups; ++r) {
                const bool cand = lane < n_groups && !kept_me;
                float v = cand ? gscore : -INFINITY;
                int gi = cand ? lane : 0x7fffffff;
                warp_argmax(v, gi);
                if (gi < n_groups) {
                    keep |= 1u << gi;
                    if (lane == gi) kept_me = true;
                }
            }
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int i = 32 * j + lane;
                if (i < N && !((keep >> (i / per_group)) & 1u)) excl |= 1u << j;
            }
        }
        int my_id = 0;
        float my_s = 0.0f;
        for (int k = 0; k < K; ++k) {
            // each lane offers its best expert still in the running (the lowest such
            // index when keys tie or are all -inf); lanes with none offer id 0x7fffffff
            float v = -INFINITY;
            int id = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int i = 32 * j + lane;
                if (!((excl >> j) & 1u) && (id == 0x7fffffff || key[j] > v)) {
                    v = key[j];
                    id = i;
                }
            }
            warp_argmax(v, id);
            // id < N: at most k < K <= (experts in the running) were taken before
            const int wl = id & 31, wj = id >> 5;
            float sv = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (j == wj) {
                    sv = s[j];
                    if (lane == wl) excl |= 1u << j;
                }
            sv = __shfl_sync(0xffffffffu, sv, wl);
            if (lane == k) {
                my_id = id;
                my_s = sv;
            }
        }
        // order the K chosen experts by id; sum their affinities in that order
        int rank = 0;
        float den = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int ok = __shfl_sync(0xffffffffu, my_id, k);
            if (lane < K && ok < my_id) ++rank;
        }
        for (int r = 0; r < K; ++r) {
            // the lane whose rank is r contributes next
            const uint32_t m = __ballot_sync(0xffffffffu, lane < K && rank == r);
            den += __shfl_sync(0xffffffffu, my_s, __ffs(m) - 1);
        }
        if (lane < K) {
            topk_idx[t * K + rank] = my_id;
            gates[t * K + rank] = __fdiv_rn(my_s, den);
            if (my_id >= 0 && my_id < N) atomicAdd(&hist[my_id], 1);
            else report(MOE_ERR_DEVICE_DATA);
        }
    }
    __syncthreads();
    if (loads)
        for (int i = threadIdx.x; i < N; i += blockDim.x)
            if (hist[i]) atomicAdd(loads + i, hist[i]);
}

template <int J>
cudaError_t launch_select(const float* zpart, int splits, int64_t T, int n_pad, const float* bias, int N, int K,
                          int n_groups, int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                          float* scores, float* logits, cudaStream_t stream) {
    const size_t smem = size_t(N) * 4 + (n_groups > 1 ? size_t(8) * N * 4 : 0);
    static PerDeviceOnce once;
    cudaError_t e = allow_smem(once, route_select_kernel<J>, 48 * 1024);
    if (e != cudaSuccess) return e;
    int64_t blocks = (T + 7) / 8;
    const int64_t cap = int64_t(num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    route_select_kernel<J><<<int(blocks), 256, smem, stream>>>(zpart, splits, T, n_pad, bias, N, K, n_groups,
                                                                topk_groups, topk_idx, gates, loads, scores,
                                                                logits);
    return cudaGetLastError();
}

}  // namespace

size_t prepared_centroid_bytes(int d, int N, int centroid_dtype) {
    const size_t terms = centroid_dtype == MOE_DTYPE_F32 ? 3 : 1;
    const size_t n_pad = size_t(N + 255) / 256 * 256;
    return (n_pad * terms * size_t(d) * 2 + 255) / 256 * 256;
}

RoutePlan plan_route(int64_t T, int d, int N, int centroid_dtype) {
    RoutePlan p{};
    p.terms = centroid_dtype == MOE_DTYPE_F32 ? 3 : 1;
    p.n_pad = (N + 255) / 256 * 256;
    const int64_t k_steps = int64_t(p.terms) * d / 64;
    const int64_t base = (T + 127) / 128 * (p.n_pad / 256);
    const int sms = num_sms();
    // Split-K count minimising (waves of tiles) x (K steps per tile) x (time of one
    // K step) + (fp32 partial logits each split writes and the selection reads back).
    // Constants: a 128 x 256 x 64 bf16 K step moves 48 KB and takes about 0.5 us on
    // one SM; partials cost 8 bytes per logit per split at about 6 TB/s.
    constexpr double kStepUs = 0.5, kBytesPerUs = 6.0e6;
    int best = 1;
    double best_cost = 1e300;
    for (int sp = 1; sp <= 64 && sp <= k_steps; ++sp) {
        if ((sp - 1) * ((k_steps + sp - 1) / sp) >= k_steps) continue;   // every split must get K steps
        const int64_t items = base * sp;
        const double waves = double((items + sms - 1) / sms);
        const double steps = double((k_steps + sp - 1) / sp);
        const double partial_us = double(sp) * double(T) * p.n_pad * 8.0 / kBytesPerUs;
        const double cost = waves * steps * kStepUs + partial_us;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = sp;
        }
    }
    p.splits = best;
    p.split_bytes = prepared_centroid_bytes(d, N, centroid_dtype);
    p.zpart_bytes = (size_t(p.splits) * size_t(T) * p.n_pad * 4 + 255) / 256 * 256;
    p.total_bytes = p.split_bytes + p.zpart_bytes;
    return p;
}

cudaError_t launch_route_prepare(const void* centroids, int centroid_dtype, int N, int d, const RoutePlan& plan,
                                 void* prepared, cudaStream_t stream) {
    const int64_t total = int64_t(plan.n_pad) * d;
    int64_t blocks = (total + 255) / 256;
    if (blocks > int64_t(num_sms()) * 16) blocks = int64_t(num_sms()) * 16;
    split_centroids_kernel<<<int(blocks), 256, 0, stream>>>(centroids, centroid_dtype == MOE_DTYPE_F32, N, plan.n_pad,
                                                            d, plan.terms, reinterpret_cast<uint16_t*>(prepared));
    return cudaGetLastError();
}

cudaError_t launch_route(const uint16_t* u, int64_t T, int d, const void* prepared, const float* bias, int N, int K,
                         int n_groups, int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                         float* scores, void* zpart_ws, const RoutePlan& plan, cudaStream_t stream, float* logits) {
    // loads may be null: the caller counts them elsewhere (the layer's permutation does)
    cudaError_t e = loads ? cudaMemsetAsync(loads, 0, sizeof(int32_t) * N, stream) : cudaSuccess;
    if (e != cudaSuccess || T == 0) return e;
    const uint16_t* esplit = reinterpret_cast<const uint16_t*>(prepared);
    float* zpart = reinterpret_cast<float*>(zpart_ws);
    CUtensorMap ta, tb;
    if (!make_kmajor_map(&ta, u, true, uint64_t(d), uint64_t(T), uint64_t(d) * 2, 128) ||
        !make_kmajor_map(&tb, esplit, true, uint64_t(plan.terms) * d, uint64_t(plan.n_pad),
                         uint64_t(plan.terms) * d * 2, 256))
        return cudaErrorInvalidValue;
    GemmArgs a{};
    a.group_offsets = nullptr;
    a.G = 1;
    a.M_total = T;
    a.Nd = plan.n_pad;
    a.Kd = plan.terms * d;
    a.k_steps = plan.terms * d / 64;
    a.a_k_repeat = plan.terms;
    a.elems_per_step = 64;
    a.splits = plan.splits;
    a.promote_steps = kBf16PromoteSteps;
    a.epilogue = MOE_EPI_F32;
    a.C = zpart;
    const int64_t items = (T + 127) / 128 * (plan.n_pad / 256) * plan.splits;
    const int grid = int(items < num_sms() ? items : num_sms());
    if ((e = run_grouped_gemm(kModeBF16, ta, tb, a, grid, stream)) != cudaSuccess) return e;

    const int Jneed = (N + 31) / 32;
    if (Jneed <= 1) return launch_select<1>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
    if (Jneed <= 2) return launch_select<2>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
    if (Jneed <= 4) return launch_select<4>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
    if (Jneed <= 8) return launch_select<8>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
    if (Jneed <= 16) return launch_select<16>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
    return launch_select<32>(zpart, plan.splits, T, plan.n_pad, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads, scores, logits, stream);
}

}  // namespace moe
