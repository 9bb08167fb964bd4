// Permutation into per-expert row blocks: the single-GPU form of the MoE
// dispatch (DeepSeek-V3 Technical Report, learn.ifs.name summary, paragraph on
// all-to-all dispatch and combine). A stable counting sort of the (token, k)
// pairs by expert: rows of expert i start at offsets[i], tokens ascending
// within an expert, and every pair keeps its row (no token is dropped).
//
//   count   warp per 32-token chunk: per-chunk expert histogram
//   scan    per expert: exclusive prefix over chunks, and the expert total
//   rank    warp per chunk: row = offsets[e] + prefix + rank among equal
//           experts in (token, k) order (__match_any_sync)
//   small   batches of at most 8192 pairs over at most 256 experts: count,
//           scan and rank in one block (one launch instead of three; the
//           decode and small layers are bound by dependent launches)
//   scatter warp per (token, 512 columns): the piece is read once and written
//           to the token's K rows (and to the shared expert's row), optionally
//           quantised to E4M3 per 1x128 tile on the way.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kChunk = 32;   // tokens per chunk

__global__ void __launch_bounds__(256) perm_count_kernel(const int32_t* __restrict__ idx, int64_t T, int N, int K,
                                                         int32_t* __restrict__ counts) {
    extern __shared__ int sh[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int* h = sh + w * N;
    const int64_t n_chunks = (T + kChunk - 1) / kChunk;
    for (int64_t c = int64_t(blockIdx.x) * 8 + w; c < n_chunks; c += int64_t(gridDim.x) * 8) {
        for (int i = lane; i < N; i += 32) h[i] = 0;
        __syncwarp();
        const int64_t p0 = c * kChunk * K, p1 = min(T, (c + 1) * kChunk) * K;
        for (int64_t p = p0 + lane; p < p1; p += 32) {
            const int e = __ldg(idx + p);
            if (e >= 0 && e < N) atomicAdd(&h[e], 1);
            else report(MOE_ERR_DEVICE_DATA);
        }
        __syncwarp();
        for (int i = lane; i < N; i += 32) counts[c * N + i] = h[i];
        __syncwarp();
    }
}

// Block b handles experts 32b..32b+31; warp s of it handles chunk segment s.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ counts, int64_t n_chunks, int N,
                                                         int32_t* __restrict__ totals, int32_t* __restrict__ loads) {
    __shared__ int part[32][33];
    const int lane = threadIdx.x & 31, seg = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const int64_t L = (n_chunks + 31) / 32;
    const int64_t c0 = seg * L, c1 = min(n_chunks, c0 + L);
    int sum = 0;
    if (e < N)
        for (int64_t c = c0; c < c1; ++c) sum += counts[c * N + e];
    part[seg][lane] = sum;
    __syncthreads();
    int run = 0;
    for (int s2 = 0; s2 < seg; ++s2) run += part[s2][lane];
    if (e < N) {
        // rewrite the counts as exclusive prefixes over the chunks
        for (int64_t c = c0; c < c1; ++c) {
            const int v = counts[c * N + e];
            counts[c * N + e] = run;
            run += v;
        }
        if (seg == 31) {
            totals[e] = run;
            if (loads) loads[e] = run;
        }
    }
}

// Exclusive scan of the expert totals into offsets (every block recomputes it).
__device__ void block_offsets(const int32_t* totals, int N, int* off_sm) {
    __shared__ int warp_tot[32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < N; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = i < N ? totals[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) warp_tot[w] = incl;
        __syncthreads();
        int before = 0;
        for (int k = 0; k < w; ++k) before += warp_tot[k];
        int all = 0;
        for (int k = 0; k < nw; ++k) all += warp_tot[k];
        if (i < N) off_sm[i] = carry + before + incl - v;
        carry += all;
        __syncthreads();
    }
    if (threadIdx.x == 0) off_sm[N] = carry;
    __syncthreads();
}

// Rows of the pairs [p0, p1), walked 32 at a time by one warp: run[e] holds
// the next row of expert e and advances past this group's pairs of e.
__device__ void rank_pairs(const int32_t* __restrict__ idx, int64_t p0, int64_t p1, int N, int K, int* run,
                           int32_t* __restrict__ perm_token, int32_t* __restrict__ dest_row) {
    const int lane = threadIdx.x & 31;
    for (int64_t pb = p0; pb < p1; pb += 32) {
        const int64_t p = pb + lane;
        const bool active = p < p1;
        int e = active ? __ldg(idx + p) : -1 - lane;
        if (e < 0 || e >= N) {
            // out of range (reported by the count pass): the pair gets no row
            if (active) dest_row[p] = -1;
            e = -1 - lane;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (active && e >= 0) {
            const int before = __popc(peers & ((1u << lane) - 1u));
            const int row = run[e] + before;
            dest_row[p] = row;
            perm_token[row] = int32_t(p / K);
        }
        __syncwarp();
        if (active && e >= 0 && (peers & ((1u << lane) - 1u)) == 0) run[e] += __popc(peers);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(256) perm_rank_kernel(const int32_t* __restrict__ idx, int64_t T, int N, int K,
                                                        const int32_t* __restrict__ prefix,
                                                        const int32_t* __restrict__ totals, int with_shared,
                                                        int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
                                                        int32_t* __restrict__ dest_row) {
    extern __shared__ int sh[];
    int* off_sm = sh;                 // [N+1]
    int* run_all = sh + N + 1;        // [8][N]
    block_offsets(totals, N, off_sm);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= N; i += blockDim.x) offsets[i] = off_sm[i];
        if (with_shared && threadIdx.x == 0) offsets[N + 1] = off_sm[N] + int32_t(T);
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int* run = run_all + w * N;
    const int64_t n_chunks = (T + kChunk - 1) / kChunk;
    for (int64_t c = int64_t(blockIdx.x) * 8 + w; c < n_chunks; c += int64_t(gridDim.x) * 8) {
        for (int i = lane; i < N; i += 32) run[i] = off_sm[i] + prefix[c * N + i];
        __syncwarp();
        rank_pairs(idx, c * kChunk * K, min(T, (c + 1) * kChunk) * K, N, K, run, perm_token, dest_row);
    }
}

// Count, scan and rank of a small batch in one block of 32 warps. Warp w owns
// the contiguous pair range [w*L, (w+1)*L), so an expert's rows still come in
// (token, k) order: warps in order, and lanes in order within a warp.
constexpr int64_t kSmallPairs = 8192;
constexpr int kSmallMaxN = 256;

__global__ void __launch_bounds__(1024) perm_small_kernel(const int32_t* __restrict__ idx, int64_t T, int N, int K,
                                                          int with_shared, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ perm_token,
                                                          int32_t* __restrict__ dest_row,
                                                          int32_t* __restrict__ loads) {
    extern __shared__ int sh[];
    int* off_sm = sh;            // [N+1]
    int* tot = sh + N + 1;       // [N]
    int* hist = tot + N;         // [32][N]: warp w's counts, then its next row per expert
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t P = T * K, L = (P + 31) / 32;
    const int64_t p0 = min(P, int64_t(w) * L), p1 = min(P, int64_t(w + 1) * L);
    for (int i = threadIdx.x; i < 32 * N; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    int* h = hist + w * N;
    for (int64_t p = p0 + lane; p < p1; p += 32) {
        const int e = __ldg(idx + p);
        if (e >= 0 && e < N) atomicAdd(&h[e], 1);
        else report(MOE_ERR_DEVICE_DATA);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int run = 0;
        for (int v = 0; v < 32; ++v) {
            const int c = hist[v * N + e];
            hist[v * N + e] = run;
            run += c;
        }
        tot[e] = run;
        if (loads) loads[e] = run;
    }
    __syncthreads();
    block_offsets(tot, N, off_sm);
    for (int i = threadIdx.x; i <= N; i += blockDim.x) offsets[i] = off_sm[i];
    if (with_shared && threadIdx.x == 0) offsets[N + 1] = off_sm[N] + int32_t(T);
    for (int i = lane; i < N; i += 32) h[i] += off_sm[i];
    __syncwarp();
    rank_pairs(idx, p0, p1, N, K, h, perm_token, dest_row);
}

// Token-major scatter of rows (bf16 copy or E4M3 1x128 quantisation). A warp
// takes one (token, 512 columns) item, 16 columns per lane (a warp per token
// walking its columns left most SMs idle in decode batches):
//   E4M3: lane l takes columns 16l..16l+15, so a 128-element tile sits in 8
//         lanes and each destination row gets one 16-byte store per lane
//         (512 contiguous bytes per warp);
//   bf16: lane l takes columns 8l..8l+7 and 256+8l..256+8l+7, so each of
//         the two 16-byte stores per destination covers 512 contiguous bytes.
template <bool kFP8>
__global__ void __launch_bounds__(256) perm_scatter_kernel(const uint16_t* __restrict__ x, int64_t T, int d, int K,
                                                           const int32_t* __restrict__ dest_row, int with_shared,
                                                           void* __restrict__ out, float* __restrict__ scales,
                                                           int64_t R) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int n_dest = K + (with_shared ? 1 : 0);
    const int off_a = kFP8 ? lane * 16 : lane * 8;    // columns of the lane's two 8-element pieces
    const int off_b = kFP8 ? lane * 16 + 8 : 256 + lane * 8;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const int steps = (d + 511) / 512;
    const int64_t items = T * steps;
    for (int64_t item = int64_t(blockIdx.x) * 8 + w; item < items; item += int64_t(gridDim.x) * 8) {
        const int64_t t = item / steps;
        const int c0 = int(item - t * steps) * 512;
        int my_dest = 0;
        if (lane < K) my_dest = __ldg(dest_row + t * K + lane);
        else if (lane == K && with_shared) my_dest = int(int64_t(T) * K + t);
        const uint16_t* src = x + t * d;
        {
            const int ca = c0 + off_a, cb = c0 + off_b;
            // d is a multiple of 128: the 8 lanes of an E4M3 tile are all active or all idle
            const bool act_a = ca < d, act_b = cb < d;
            const uint4 v0 = act_a ? __ldg(reinterpret_cast<const uint4*>(src + ca)) : zero;
            const uint4 v1 = act_b ? __ldg(reinterpret_cast<const uint4*>(src + cb)) : zero;
            if constexpr (!kFP8) {
                for (int k = 0; k < n_dest; ++k) {
                    const int row = __shfl_sync(0xffffffffu, my_dest, k);
                    // rows outside [0, R) come from out-of-range expert ids: skipped
                    if (row >= 0 && row < R) {
                        uint16_t* dst = reinterpret_cast<uint16_t*>(out) + int64_t(row) * d;
                        if (act_a) *reinterpret_cast<uint4*>(dst + ca) = v0;
                        if (act_b) *reinterpret_cast<uint4*>(dst + cb) = v1;
                    }
                }
            } else {
                const uint32_t in[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(in[i])), fabsf(bf16_hi(in[i]))));
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sc = tile_scale(amax);
                uint32_t q[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q[i] = pack_e4m3x2(__fdiv_rn(bf16_lo(in[2 * i]), sc), __fdiv_rn(bf16_hi(in[2 * i]), sc)) |
                           (pack_e4m3x2(__fdiv_rn(bf16_lo(in[2 * i + 1]), sc), __fdiv_rn(bf16_hi(in[2 * i + 1]), sc))
                            << 16);
                const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                const int kb = ca / 128;
                for (int k = 0; k < n_dest; ++k) {
                    const int row = __shfl_sync(0xffffffffu, my_dest, k);
                    if (act_a && row >= 0 && row < R) {
                        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) + int64_t(row) * d + ca) = qv;
                        if ((lane & 7) == 0) scales[int64_t(kb) * R + row] = sc;
                    }
                }
            }
        }
    }
}

}  // namespace

size_t permute_ws_bytes(int64_t T, int N) {
    const int64_t n_chunks = (T + kChunk - 1) / kChunk;
    return (size_t(n_chunks) * N * 4 + size_t(N) * 4 + 255) / 256 * 256;
}

cudaError_t launch_permute(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K, int out_dtype,
                           int with_shared, int32_t* offsets, int32_t* perm_token, int32_t* dest_row, void* x_perm,
                           float* x_perm_scales, void* ws, cudaStream_t stream, int32_t* loads) {
    const int64_t n_chunks = (T + kChunk - 1) / kChunk;
    int32_t* counts = reinterpret_cast<int32_t*>(ws);
    int32_t* totals = counts + n_chunks * N;
    cudaError_t e;
    const int64_t cap = int64_t(num_sms()) * 8;
    if (T == 0) {
        if ((e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (N + 1 + (with_shared ? 1 : 0)), stream)) != cudaSuccess)
            return e;
        return loads ? cudaMemsetAsync(loads, 0, sizeof(int32_t) * N, stream) : cudaSuccess;
    }
    if (T * K <= kSmallPairs && N <= kSmallMaxN) {
        perm_small_kernel<<<1, 1024, size_t(34 * N + 1) * 4, stream>>>(topk_idx, T, N, K, with_shared, offsets,
                                                                       perm_token, dest_row, loads);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
        {
            int64_t blocks = (n_chunks + 7) / 8;
            if (blocks > cap) blocks = cap;
            perm_count_kernel<<<int(blocks), 256, size_t(8) * N * 4, stream>>>(topk_idx, T, N, K, counts);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        perm_scan_kernel<<<(N + 31) / 32, 1024, 0, stream>>>(counts, n_chunks, N, totals, loads);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        int64_t blocks = (n_chunks + 7) / 8;
        if (blocks > cap) blocks = cap;
        const size_t smem = size_t(N + 1) * 4 + size_t(8) * N * 4;
        static PerDeviceOnce once;
        if ((e = allow_smem(once, perm_rank_kernel, 64 * 1024)) != cudaSuccess) return e;
        perm_rank_kernel<<<int(blocks), 256, smem, stream>>>(topk_idx, T, N, K, counts, totals, with_shared, offsets,
                                                             perm_token, dest_row);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (x_perm) {   // null: the rows are not moved (the grouped GEMM gathers them)
        const int64_t R = T * K + (with_shared ? T : 0);
        int64_t blocks = (T * ((d + 511) / 512) + 7) / 8;   // a warp per (token, 512 columns)
        if (blocks > cap * 2) blocks = cap * 2;
        if (out_dtype == MOE_DTYPE_E4M3)
            perm_scatter_kernel<true><<<int(blocks), 256, 0, stream>>>(x, T, d, K, dest_row, with_shared, x_perm,
                                                                       x_perm_scales, R);
        else
            perm_scatter_kernel<false><<<int(blocks), 256, 0, stream>>>(x, T, d, K, dest_row, with_shared, x_perm,
                                                                        nullptr, R);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
