// The layer's backward pass and training step: the memory-bound kernels.
//
// Sources (the DeepSeek-V3 Technical Report as summarised on the web):
//   nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)", "The
//   notation" (the layer formula h'_t = u_t + FFN_shared(u_t) +
//   sum_k g_{t,k} FFN_{idx}(u_t)) and "The idea", FP8-training item (the heavy
//   products of training run in FP8 with tile and block scales);
//   learn.ifs.name "DeepSeek-V3 Technical Report", FP8 paragraph (1x128 tiles,
//   128x128 blocks) and bias paragraph (the bias moves after each step).
// Readings: the gradient of the layer formula with the expert choice held
// fixed; every quantisation and bf16 rounding passed straight through; each
// backward product takes FP8 operands scaled along its own contraction
// dimension (a weight gradient contracts over an expert's tokens, so its
// operands get one scale per 128 tokens and column).
//
// Kernels (rows r index the forward's permuted rows: routed rows grouped by
// expert, then T rows of the shared expert):
//   combine_bwd     one warp per (token, row): dg_{t,k} = G_t . y_{row(t,k)} and
//                   the dgrad operand dY = g G_t per 1x128 tile (G_t's codes, g
//                   times its scales)
//   swiglu_bwd      one half-warp per (row, 128 outputs): dH from the stored
//                   bf16 H and dA, stored in bf16 and quantised per 1x128 tile
//   kblock_offsets  each group's first 128-row block in the padded K layout
//   pad_rows        the permuted row of every padded row of that layout
//   quant_t         the weight-gradient operands: 128 rows x 512 columns per
//                   block (a cp.async ring of 64-column chunks), transposed,
//                   one scale per (128 rows, column)
//   unpermute_bwd   one block per token: gate backward and du
//   centroid_grad   de_i = sum over expert i's rows of dz u_t, in row order
//   fp8_transpose   128x128 E4M3 blocks transposed with their scales
//   sgd_requant     w <- fl32(w - fl32(lr g)) on fp32 masters, then the
//                   128x128 quantisation, stored as is and transposed
// All HBM bound; every sum runs in a fixed order (results reproducible bit for bit).
#include "common.cuh"
#include "e4m3.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf16_lo(v.x);
    f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y);
    f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z);
    f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w);
    f[7] = bf16_hi(v.w);
}

// 8 values of one 1x128 tile (16 lanes hold a tile) -> 8 codes; returns the scale.
__device__ __forceinline__ float quant8_tile16(const float (&f)[8], uint2& codes) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = tile_scale(amax);
    codes.x = pack_e4m3x2(__fdiv_rn(f[0], sc), __fdiv_rn(f[1], sc)) |
              (pack_e4m3x2(__fdiv_rn(f[2], sc), __fdiv_rn(f[3], sc)) << 16);
    codes.y = pack_e4m3x2(__fdiv_rn(f[4], sc), __fdiv_rn(f[5], sc)) |
              (pack_e4m3x2(__fdiv_rn(f[6], sc), __fdiv_rn(f[7], sc)) << 16);
    return sc;
}

constexpr int kMaxK = 16;

// One block of 32 (K + 1) threads per token t: warp k < K takes the routed row
// of (t, k) -- dg_{t,k} = G_t . y_row and the row's dgrad operand -- and warp
// K the shared expert's row. Lanes hold 8 consecutive columns; a 1x128 tile
// is a half-warp, and a warp steps over d 256 columns at a time.
// The dgrad operand of a routed row is the tile rule applied to g G_t: the
// rule is scale-invariant (amax and every value scale by g), so its codes are
// those of G_t's tile and its scale is g times G_t's. The block quantises G_t
// once (its warps share the steps) into shared memory, and every warp copies
// the codes to its row.
__global__ void __launch_bounds__(32 * (kMaxK + 1)) combine_bwd_kernel(
    const uint16_t* __restrict__ G, const uint16_t* __restrict__ y, const float* __restrict__ gates,
    const int32_t* __restrict__ dest, int64_t T, int d, int K, int64_t R, uint8_t* __restrict__ qdy,
    float* __restrict__ sdy, float* __restrict__ row_gate, float* __restrict__ dg) {
    extern __shared__ __align__(16) uint8_t cb_smem[];
    uint2* codes_sm = reinterpret_cast<uint2*>(cb_smem);               // [d / 8]: G_t's codes
    float* scale_sm = reinterpret_cast<float*>(cb_smem + d);           // [d / 128]: its tile scales
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x & 31, k = threadIdx.x >> 5;
    const bool routed = k < K;
    const int64_t row = routed ? int64_t(__ldg(dest + t * K + k)) : T * K + t;
    const float g = routed ? __ldg(gates + t * K + k) : 1.0f;
    const uint4* Gp = reinterpret_cast<const uint4*>(G + t * d);
    const uint4* yp = reinterpret_cast<const uint4*>(y + row * d);
    // d % 256 == 0 (the layer's rule): every lane of a warp runs each step, as the
    // shuffles of the tile's amax require
    const int steps = d / 256;
    for (int st = k; st < steps; st += K + 1) {   // warp-uniform
        const int c = lane + 32 * st;
        float gv[8];
        unpack8(__ldg(Gp + c), gv);
        uint2 codes;
        const float sc = quant8_tile16(gv, codes);
        codes_sm[c] = codes;
        if ((lane & 15) == 0) scale_sm[c / 16] = sc;
    }
    __syncthreads();
    float acc = 0.0f;
    // Two steps' loads are issued before either is used (bytes in flight for HBM);
    // the dot product keeps its step order.
    constexpr int kU = 2;
    for (int s0 = 0; s0 < steps; s0 += kU) {
        uint4 gr[kU], yr[kU];
        if (routed) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (s0 + u < steps) {
                    const int c = lane + 32 * (s0 + u);
                    gr[u] = __ldg(Gp + c);
                    yr[u] = __ldg(yp + c);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (s0 + u < steps) {
                const int c = lane + 32 * (s0 + u);
                if (routed) {
                    float gv[8], yv[8];
                    unpack8(gr[u], gv);
                    unpack8(yr[u], yv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc = fmaf(gv[i], yv[i], acc);
                }
                *reinterpret_cast<uint2*>(qdy + row * d + int64_t(c) * 8) = codes_sm[c];
                if ((lane & 15) == 0) {
                    const float sc = scale_sm[c / 16];
                    sdy[(int64_t(c) / 16) * R + row] = routed ? __fmul_rn(g, sc) : sc;
                }
            }
        }
    }
    if (routed) {
        // a fixed xor tree over the warp's partial sums
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            dg[t * K + k] = acc;
            row_gate[row] = g;
        }
    } else if (lane == 0) {
        row_gate[row] = 1.0f;
    }
}

// One half-warp per (row r, pair p of 128-column blocks): lanes hold 8 of the
// 128 outputs (16-byte loads and stores). H's columns 256p.. are the gate
// products, 256p+128.. the up ones. The two halves of a warp take consecutive
// items; a half past the last item computes on zeros and stores nothing (the
// amax shuffles stay inside a half).
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const uint16_t* __restrict__ dA,
                                                         const uint16_t* __restrict__ H, int64_t R, int I,
                                                         uint16_t* __restrict__ dH, uint8_t* __restrict__ qdh,
                                                         float* __restrict__ sdh) {
    const int hl = threadIdx.x & 15;
    const int pairs = I / 128;
    const int64_t item = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
    const bool active = item < R * pairs;
    const int64_t r = active ? item / pairs : 0;
    const int p = active ? int(item - r * pairs) : 0;
    const int I2 = 2 * I;
    uint4 va = make_uint4(0u, 0u, 0u, 0u), v1 = va, v3 = va;
    if (active) {
        va = __ldg(reinterpret_cast<const uint4*>(dA + r * I + 128 * p) + hl);
        v1 = __ldg(reinterpret_cast<const uint4*>(H + r * I2 + 256 * p) + hl);
        v3 = __ldg(reinterpret_cast<const uint4*>(H + r * I2 + 256 * p + 128) + hl);
    }
    float a[8], h1[8], h3[8];
    unpack8(va, a);
    unpack8(v1, h1);
    unpack8(v3, h3);
    float d1[8], d3[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float sg = sigmoid_f(h1[i]);
        d1[i] = a[i] * h3[i] * sg * (1.0f + h1[i] * (1.0f - sg));
        d3[i] = a[i] * h1[i] * sg;
    }
    // stored in bf16; the quantisation below reads the stored values
    const uint4 b1 = make_uint4(pack_bf16x2(d1[0], d1[1]), pack_bf16x2(d1[2], d1[3]), pack_bf16x2(d1[4], d1[5]),
                                pack_bf16x2(d1[6], d1[7]));
    const uint4 b3 = make_uint4(pack_bf16x2(d3[0], d3[1]), pack_bf16x2(d3[2], d3[3]), pack_bf16x2(d3[4], d3[5]),
                                pack_bf16x2(d3[6], d3[7]));
    if (active) {
        reinterpret_cast<uint4*>(dH + r * I2 + 256 * p)[hl] = b1;
        reinterpret_cast<uint4*>(dH + r * I2 + 256 * p + 128)[hl] = b3;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float f[8];
        unpack8(half ? b3 : b1, f);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = tile_scale(amax);
        const uint2 q = make_uint2(pack_e4m3x2(__fdiv_rn(f[0], sc), __fdiv_rn(f[1], sc)) |
                                       (pack_e4m3x2(__fdiv_rn(f[2], sc), __fdiv_rn(f[3], sc)) << 16),
                                   pack_e4m3x2(__fdiv_rn(f[4], sc), __fdiv_rn(f[5], sc)) |
                                       (pack_e4m3x2(__fdiv_rn(f[6], sc), __fdiv_rn(f[7], sc)) << 16));
        if (active) {
            reinterpret_cast<uint2*>(qdh + r * I2 + 256 * p + 128 * half)[hl] = q;
            if (hl == 0) sdh[int64_t(2 * p + half) * R + r] = sc;
        }
    }
}

// kofs[g] = sum over g' < g of ceil(rows_g' / 128): one warp.
__global__ void kblock_offsets_kernel(const int32_t* __restrict__ offsets, int G, int32_t* __restrict__ kofs) {
    const int lane = threadIdx.x;
    int running = 0;
    for (int base = 0; base <= G; base += 32) {
        const int g = base + lane;
        int blocks = 0;
        if (g < G) {
            const int n = offsets[g + 1] - offsets[g];
            blocks = n > 0 ? (n + 127) / 128 : 0;
        }
        int incl = blocks;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (g <= G) kofs[g] = running + incl - blocks;
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// prow[p] = the permuted row at padded row p of the weight-gradient K layout
// (group g's rows start at 128 kofs[g]), or -1 for padding: one thread per padded row.
__global__ void __launch_bounds__(256) pad_rows_kernel(const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ kofs, int G, int64_t Kp,
                                                       int32_t* __restrict__ prow) {
    const int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p >= Kp) return;
    const int b = int(p >> 7);
    int r = -1;
    if (b < kofs[G]) {
        int lo = 0, hi = G;   // the last g with kofs[g] <= b
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (kofs[mid] <= b) lo = mid;
            else hi = mid;
        }
        const int64_t rr = offsets[lo] + int64_t(b - kofs[lo]) * 128 + (p & 127);
        if (rr < offsets[lo + 1]) r = int(rr);
    }
    prow[p] = r;
}

enum { kSrcScaledG = 0, kSrcTokens = 1, kSrcRows = 2, kSrcSwiglu = 3 };

struct QuantTArgs {
    const int32_t* prow;        // [Kp] permuted row of each padded row, -1 for padding
    const int32_t* kofs;        // [G+1] the groups' 128-row block offsets (padded)
    int G;
    int64_t TK;                 // routed rows; row r >= TK is token r - TK (shared expert)
    const int32_t* perm_token;  // [TK]
    const float* row_gate;      // kSrcScaledG: g of each row
    const uint16_t* src;        // G / u [T, C]; dH [R, C]; H [R, 2C]
    int C;                      // output rows (columns of the source operand)
    int64_t Kp;                 // padded rows (row stride of q)
    uint8_t* q;                 // [C][Kp]
    float* s;                   // [Kp/128][C]
};

constexpr int kQtStages = 3;                // 64-column chunks in shared memory per block
constexpr int kQtChunks = 8;                // chunks per block
constexpr int kQtChunkBytes = 128 * 128;    // 128 rows x 64 bf16 columns

template <int kSrc>
__host__ __device__ constexpr int qt_sources() {   // SwiGLU: the gate and the up products
    return kSrc == kSrcSwiglu ? 2 : 1;
}
template <int kSrc>
__host__ __device__ constexpr int qt_smem_bytes() {
    return kQtStages * qt_sources<kSrc>() * kQtChunkBytes;
}

// One block per (128-row block b of the padded layout, 8 chunks of 64
// columns). The block looks its 128 source rows up once, then streams the
// chunks through a 3-stage cp.async ring: while it quantises chunk j, chunks
// j+1 and j+2 are in flight. Per chunk and column: the amax of the column's 128
// rows, the scale and the codes, written transposed. Row blocks are adjacent in
// the grid, so the blocks running side by side write adjacent 128-byte pieces
// of each output row.
// Shared layout of a chunk: row r's 128 bytes as eight 16-byte pieces, piece k
// at place k ^ (r / 16 % 8). A thread of the quantisation reads one 32-bit
// word (two columns) of 16 rows, 16 rows apart from its neighbours: with the
// swizzle the 32 lanes of a warp hit 32 banks.
template <int kSrc>
__global__ void __launch_bounds__(256) quant_t_kernel(const QuantTArgs a) {
    constexpr int kL = qt_sources<kSrc>();
    extern __shared__ __align__(128) uint8_t qt_ring[];   // [kQtStages][kL][128 rows][128 bytes]
    __shared__ int row_src[128];
    __shared__ float row_w[128];
    const int64_t b = blockIdx.x;
    const int tid = threadIdx.x;
    if (b >= a.kofs[a.G]) return;   // block-uniform: K blocks past the last group are never read
    const int j0 = int(blockIdx.y) * kQtChunks;
    const int nj = min(kQtChunks, a.C / 64 - j0);
    if (tid < 128) {
        const int r = a.prow[b * 128 + tid];
        int srow = -1;
        float wgt = 0.0f;
        if (r >= 0) {
            if (kSrc == kSrcScaledG || kSrc == kSrcTokens) srow = r < a.TK ? a.perm_token[r] : int(r - a.TK);
            else srow = r;
            if (kSrc == kSrcScaledG) wgt = a.row_gate[r];
        }
        row_src[tid] = srow;
        row_w[tid] = wgt;
    }
    __syncthreads();
    const uint32_t ring = smem_u32(qt_ring);
    // copies: a thread moves piece k of rows rr, rr + 32, rr + 64, rr + 96 (padding rows: zeros)
    const int k = tid & 7, rr = tid >> 3;
    auto issue = [&](int j) {
        const uint32_t st = ring + uint32_t((j % kQtStages) * kL * kQtChunkBytes);
        const int c = (j0 + j) * 64 + 8 * k;   // the piece's first column
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = rr + 32 * i;
            const int sr = row_src[r];
            const int64_t srow = sr >= 0 ? sr : 0;
            const uint32_t place = uint32_t(r) * 128u + uint32_t((k ^ ((r >> 4) & 7)) * 16);
#pragma unroll
            for (int l = 0; l < kL; ++l) {
                // SwiGLU: output column c reads the gate product at 256 (c / 128) + c % 128
                // and the up product 128 further
                const uint16_t* src = kSrc == kSrcSwiglu
                                          ? a.src + srow * (2 * a.C) + 256 * (c / 128) + (c % 128) + 128 * l
                                          : a.src + srow * a.C + c;
                cp_async_16z(st + uint32_t(l * kQtChunkBytes) + place, src, sr >= 0 ? 16u : 0u);
            }
        }
    };
#pragma unroll
    for (int j = 0; j < kQtStages - 1; ++j) {
        if (j < nj) issue(j);
        cp_async_commit();
    }
    // quantisation: a thread takes columns 2 cp, 2 cp + 1 of rows 16 qt .. 16 qt + 15
    const int qt = tid & 7, cp = tid >> 3;
    for (int j = 0; j < nj; ++j) {
        cp_async_wait_group<kQtStages - 2>();   // this thread's copies of chunk j have landed
        __syncthreads();                        // ... and every thread's; chunk j - 1 is read
        if (j + kQtStages - 1 < nj) issue(j + kQtStages - 1);
        cp_async_commit();
        const uint8_t* st = qt_ring + (j % kQtStages) * kL * kQtChunkBytes;
        const int word = (((cp >> 2) ^ qt) * 16) + (cp & 3) * 4;   // rows 16 qt..: r / 16 % 8 = qt
        float v0[16], v1[16];
        float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * qt + i;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(st + r * 128 + word);
            if (kSrc == kSrcSwiglu) {
                const uint32_t w3 = *reinterpret_cast<const uint32_t*>(st + kQtChunkBytes + r * 128 + word);
                const float g0 = bf16_lo(w), g1 = bf16_hi(w);
                v0[i] = g0 * sigmoid_f(g0) * bf16_lo(w3);
                v1[i] = g1 * sigmoid_f(g1) * bf16_hi(w3);
            } else if (kSrc == kSrcScaledG) {
                const float wg = row_w[r];
                v0[i] = wg * bf16_lo(w);
                v1[i] = wg * bf16_hi(w);
            } else {
                v0[i] = bf16_lo(w);
                v1[i] = bf16_hi(w);
            }
            am0 = fmaxf(am0, fabsf(v0[i]));
            am1 = fmaxf(am1, fabsf(v1[i]));
        }
        // the 8 lanes of a column pair: lane bits 0-2
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            am0 = fmaxf(am0, __shfl_xor_sync(0xffffffffu, am0, o));
            am1 = fmaxf(am1, __shfl_xor_sync(0xffffffffu, am1, o));
        }
        const float sc0 = tile_scale(am0), sc1 = tile_scale(am1);
        // the quotients by reciprocal where that cannot change a code (e4m3_quotient): with
        // IEEE divisions alone this kernel was bound by them (2.6 ms against 1.7 ms at the
        // V3 training shape)
        const float r0 = e4m3_recip(sc0), r1 = e4m3_recip(sc1);
        uint32_t q0[4], q1[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            q0[m] = pack_e4m3x2(e4m3_quotient(v0[4 * m], sc0, r0), e4m3_quotient(v0[4 * m + 1], sc0, r0)) |
                    (pack_e4m3x2(e4m3_quotient(v0[4 * m + 2], sc0, r0), e4m3_quotient(v0[4 * m + 3], sc0, r0))
                     << 16);
            q1[m] = pack_e4m3x2(e4m3_quotient(v1[4 * m], sc1, r1), e4m3_quotient(v1[4 * m + 1], sc1, r1)) |
                    (pack_e4m3x2(e4m3_quotient(v1[4 * m + 2], sc1, r1), e4m3_quotient(v1[4 * m + 3], sc1, r1))
                     << 16);
        }
        const int col = (j0 + j) * 64 + 2 * cp;
        uint8_t* dst = a.q + int64_t(col) * a.Kp + b * 128 + 16 * qt;
        *reinterpret_cast<uint4*>(dst) = make_uint4(q0[0], q0[1], q0[2], q0[3]);
        *reinterpret_cast<uint4*>(dst + a.Kp) = make_uint4(q1[0], q1[1], q1[2], q1[3]);
        if (qt == 0) {
            a.s[b * a.C + col] = sc0;
            a.s[b * a.C + col + 1] = sc1;
        }
    }
}

// One block of 256 threads per token: the gate backward (K scalars, thread 0)
// and du_t = G_t + dX_shared,t + sum_k dX_row(t,k) + sum_k dz_k e_idx(t,k).
__global__ void __launch_bounds__(256) unpermute_bwd_kernel(
    const uint16_t* __restrict__ G, const uint16_t* __restrict__ dX, const int32_t* __restrict__ dest,
    const int32_t* __restrict__ topk, const float* __restrict__ gates, const float* __restrict__ scores,
    const float* __restrict__ logits, const float* __restrict__ dg, const void* __restrict__ centroids,
    int centroid_f32, int64_t T, int d, int N,
    int K, uint16_t* __restrict__ du, float* __restrict__ dz_row, float* __restrict__ dz_out) {
    __shared__ float dz[kMaxK];
    __shared__ int64_t rows[kMaxK];
    __shared__ int ids[kMaxK];
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) {
        float S = 0.0f, c = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int e = topk[t * K + k];
            ids[k] = e;
            rows[k] = dest[t * K + k];
            S += scores[t * N + e];
            c = fmaf(gates[t * K + k], dg[t * K + k], c);
        }
        for (int k = 0; k < K; ++k) {
            // s'(z) = s (1 - s) from the logit: e^-|z| / (1 + e^-|z|)^2, accurate where s is near 1
            const float ez = expf(-fabsf(logits[t * N + ids[k]]));
            const float dsig = __fdiv_rn(ez, (1.0f + ez) * (1.0f + ez));
            const float v = __fdiv_rn(dg[t * K + k] - c, S) * dsig;
            dz[k] = v;
            dz_row[rows[k]] = v;
            if (dz_out) dz_out[t * K + k] = v;
        }
    }
    __syncthreads();
    const int64_t shared_row = T * K + t;
    for (int c = tid; c < d / 8; c += 256) {
        float acc[8], f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(G + t * d) + c), acc);
        unpack8(__ldg(reinterpret_cast<const uint4*>(dX + shared_row * d) + c), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += f[j];
        for (int k = 0; k < K; ++k) {
            unpack8(__ldg(reinterpret_cast<const uint4*>(dX + rows[k] * d) + c), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += f[j];
        }
        for (int k = 0; k < K; ++k) {
            const int64_t e = ids[k];
            if (centroid_f32) {
                const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(centroids) + e * d) + 2 * c;
                const float4 x0 = __ldg(p), x1 = __ldg(p + 1);
                const float ev[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(dz[k], ev[j], acc[j]);
            } else {
                unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(centroids) + e * d) + c), f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(dz[k], f[j], acc[j]);
            }
        }
        reinterpret_cast<uint4*>(du + t * d)[c] =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
    }
}

// Block (expert i, 256 columns): de[i, cols] = sum over the expert's rows r of
// dz_row[r] * u[token(r), cols]. Warp w takes the rows r0 + w, r0 + w + 8, ...
// (lane: 8 columns), then the 8 warps' sums are added in warp order: a fixed
// order, so the result is reproducible.
__global__ void __launch_bounds__(256) centroid_grad_kernel(const uint16_t* __restrict__ u,
                                                            const int32_t* __restrict__ offsets,
                                                            const int32_t* __restrict__ perm_token,
                                                            const float* __restrict__ dz_row, int d,
                                                            float* __restrict__ de) {
    __shared__ float part[8][256];
    const int i = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c0 = blockIdx.y * 256;
    const int col = c0 + lane * 8;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int r0 = offsets[i], r1 = offsets[i + 1];
    if (col < d) {
        for (int r = r0 + w; r < r1; r += 8) {
            const float wt = __ldg(dz_row + r);
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(u + int64_t(__ldg(perm_token + r)) * d + col)), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = fmaf(wt, f[j], acc[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) part[w][lane * 8 + j] = acc[j];
    __syncthreads();
    const int c = c0 + threadIdx.x;
    if (c < d) {
        float v = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) v += part[k][threadIdx.x];
        de[int64_t(i) * d + c] = v;
    }
}

// One block per (group, 128x128 block): codes transposed through shared memory.
__global__ void __launch_bounds__(256) fp8_transpose_kernel(const uint8_t* __restrict__ q, const float* __restrict__ s,
                                                            int rows, int cols, uint8_t* __restrict__ qt,
                                                            float* __restrict__ st) {
    __shared__ uint8_t tile[128][129];
    const int bc = blockIdx.x, br = blockIdx.y;
    const int64_t g = blockIdx.z;
    const int tid = threadIdx.x;
    const uint8_t* src = q + g * rows * int64_t(cols);
    uint8_t* dst = qt + g * rows * int64_t(cols);
    // read: 8 lanes per row of 128 bytes (16 each), 32 rows per pass
    for (int r = tid >> 3; r < 128; r += 32) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + int64_t(br * 128 + r) * cols + bc * 128) + (tid & 7));
        const uint8_t* bv = reinterpret_cast<const uint8_t*>(&v);
#pragma unroll
        for (int j = 0; j < 16; ++j) tile[r][(tid & 7) * 16 + j] = bv[j];
    }
    __syncthreads();
    for (int r = tid >> 3; r < 128; r += 32) {
        uint4 v;
        uint8_t* bv = reinterpret_cast<uint8_t*>(&v);
#pragma unroll
        for (int j = 0; j < 16; ++j) bv[j] = tile[(tid & 7) * 16 + j][r];
        reinterpret_cast<uint4*>(dst + int64_t(bc * 128 + r) * rows + br * 128)[tid & 7] = v;
    }
    if (tid == 0) {
        const int nbr = rows / 128, nbc = cols / 128;
        st[g * nbr * nbc + int64_t(bc) * nbr + br] = s[g * nbr * nbc + int64_t(br) * nbc + bc];
    }
}

// One block per (group, 128x128 block) of an fp32 master [G][rows][cols]:
// w <- fl32(w - fl32(lr * grad)), then the block's scale amax/448 and codes,
// stored row-major (q, s [G][rows/128][cols/128]) and transposed (qt [G][cols][rows],
// st [G][cols/128][rows/128]). Warp w takes rows 16w..16w+15 of the block and
// lane l columns 4l..4l+3, so every load and store of a warp covers one whole
// 512-byte row of the block. The first pass updates the master and takes the
// amax; the second reads the new values back (from L2) to quantise them, so a
// thread never holds more than 4 rows (more blocks per SM, more loads in flight).
__global__ void __launch_bounds__(256, 4) sgd_requant_kernel(float* __restrict__ w, const float* __restrict__ grad,
                                                          int rows, int cols, float lr, uint8_t* __restrict__ q,
                                                          float* __restrict__ s, uint8_t* __restrict__ qt,
                                                          float* __restrict__ st) {
    __shared__ uint8_t tile[128][132];
    __shared__ float warp_max[8];
    const int bc = blockIdx.x, br = blockIdx.y;
    const int64_t g = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
    const int64_t base = g * int64_t(rows) * cols + int64_t(br * 128 + 16 * wp) * cols + bc * 128 + 4 * lane;
    float amax = 0.0f;
#pragma unroll
    for (int i0 = 0; i0 < 16; i0 += 4) {
        float4 v[4];
        float4 d[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t off = base + int64_t(i0 + i) * cols;
            v[i] = *reinterpret_cast<const float4*>(w + off);
            d[i] = __ldg(reinterpret_cast<const float4*>(grad + off));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // two fp32 roundings, never fused: the product, then the difference
            v[i].x = __fsub_rn(v[i].x, __fmul_rn(lr, d[i].x));
            v[i].y = __fsub_rn(v[i].y, __fmul_rn(lr, d[i].y));
            v[i].z = __fsub_rn(v[i].z, __fmul_rn(lr, d[i].z));
            v[i].w = __fsub_rn(v[i].w, __fmul_rn(lr, d[i].w));
            *reinterpret_cast<float4*>(w + base + int64_t(i0 + i) * cols) = v[i];
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_max[wp] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float sc = tile_scale(amax);
#pragma unroll
    for (int i0 = 0; i0 < 16; i0 += 4) {
        float4 x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = *reinterpret_cast<const float4*>(w + base + int64_t(i0 + i) * cols);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = pack_e4m3x2(__fdiv_rn(x[i].x, sc), __fdiv_rn(x[i].y, sc)) |
                               (pack_e4m3x2(__fdiv_rn(x[i].z, sc), __fdiv_rn(x[i].w, sc)) << 16);
            *reinterpret_cast<uint32_t*>(q + base + int64_t(i0 + i) * cols) = c;
            *reinterpret_cast<uint32_t*>(&tile[16 * wp + i0 + i][4 * lane]) = c;
        }
    }
    __syncthreads();
    // transposed: 8 lanes per output row of 128 bytes (16 each), 32 rows per pass
    uint8_t* dst = qt + g * int64_t(rows) * cols;
    for (int c = tid >> 3; c < 128; c += 32) {
        uint4 v;
        uint8_t* bv = reinterpret_cast<uint8_t*>(&v);
#pragma unroll
        for (int j = 0; j < 16; ++j) bv[j] = tile[(tid & 7) * 16 + j][c];
        reinterpret_cast<uint4*>(dst + int64_t(bc * 128 + c) * rows + br * 128)[tid & 7] = v;
    }
    if (tid == 0) {
        const int nbr = rows / 128, nbc = cols / 128;
        s[g * nbr * nbc + int64_t(br) * nbc + bc] = sc;
        st[g * nbr * nbc + int64_t(bc) * nbr + br] = sc;
    }
}

__global__ void __launch_bounds__(256) sgd_f32_kernel(float* __restrict__ w, const float* __restrict__ grad, int64_t n,
                                                      float lr) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        w[i] = __fsub_rn(w[i], __fmul_rn(lr, __ldg(grad + i)));
}

int grid_for(int64_t items, int per_block) {
    int64_t b = (items + per_block - 1) / per_block;
    const int64_t cap = int64_t(num_sms()) * 16;
    return int(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_combine_bwd(const uint16_t* G, const uint16_t* y, const float* gates, const int32_t* dest,
                               int64_t T, int d, int K, int64_t R, uint8_t* qdy, float* sdy, float* row_gate,
                               float* dg, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int smem = d + d / 32;   // G_t's codes and tile scales
    static PerDeviceOnce once;
    cudaError_t e = allow_smem(once, combine_bwd_kernel, 227 * 1024);
    if (e != cudaSuccess) return e;
    combine_bwd_kernel<<<unsigned(T), 32 * (K + 1), smem, stream>>>(G, y, gates, dest, T, d, K, R, qdy, sdy,
                                                                    row_gate, dg);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const uint16_t* dA, const uint16_t* H, int64_t R, int I, uint16_t* dH, uint8_t* qdh,
                              float* sdh, cudaStream_t stream) {
    const int64_t items = R * (I / 128);   // a half-warp each, 16 per block
    if (items == 0) return cudaSuccess;
    swiglu_bwd_kernel<<<unsigned((items + 15) / 16), 256, 0, stream>>>(dA, H, R, I, dH, qdh, sdh);
    return cudaGetLastError();
}

cudaError_t launch_kblock_offsets(const int32_t* offsets, int G, int32_t* kofs, cudaStream_t stream) {
    kblock_offsets_kernel<<<1, 32, 0, stream>>>(offsets, G, kofs);
    return cudaGetLastError();
}

cudaError_t launch_pad_rows(const int32_t* offsets, const int32_t* kofs, int G, int64_t Kp, int32_t* prow,
                            cudaStream_t stream) {
    if (Kp == 0) return cudaSuccess;
    pad_rows_kernel<<<unsigned((Kp + 255) / 256), 256, 0, stream>>>(offsets, kofs, G, Kp, prow);
    return cudaGetLastError();
}

cudaError_t launch_quant_t(int src_kind, const int32_t* prow, const int32_t* kofs, int G, int64_t TK,
                           const int32_t* perm_token, const float* row_gate, const uint16_t* src, int C,
                           int64_t Kp, uint8_t* q, float* s, cudaStream_t stream) {
    QuantTArgs a{prow, kofs, G, TK, perm_token, row_gate, src, C, Kp, q, s};
    const dim3 grid(unsigned(Kp / 128), unsigned((C / 64 + kQtChunks - 1) / kQtChunks));
    if (grid.x == 0 || C == 0) return cudaSuccess;
    cudaError_t e;
    auto run = [&](auto kernel, int bytes, PerDeviceOnce& once) {
        if ((e = allow_smem(once, kernel, bytes)) != cudaSuccess) return e;
        kernel<<<grid, 256, bytes, stream>>>(a);
        return cudaGetLastError();
    };
    static PerDeviceOnce o0, o1, o2, o3;
    switch (src_kind) {
        case kSrcScaledG: return run(quant_t_kernel<kSrcScaledG>, qt_smem_bytes<kSrcScaledG>(), o0);
        case kSrcTokens: return run(quant_t_kernel<kSrcTokens>, qt_smem_bytes<kSrcTokens>(), o1);
        case kSrcRows: return run(quant_t_kernel<kSrcRows>, qt_smem_bytes<kSrcRows>(), o2);
        case kSrcSwiglu: return run(quant_t_kernel<kSrcSwiglu>, qt_smem_bytes<kSrcSwiglu>(), o3);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_unpermute_bwd(const uint16_t* G, const uint16_t* dX, const int32_t* dest, const int32_t* topk,
                                 const float* gates, const float* scores, const float* logits, const float* dg,
                                 const void* centroids, int centroid_f32, int64_t T, int d, int N, int K, uint16_t* du,
                                 float* dz_row, float* dz_out, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    unpermute_bwd_kernel<<<unsigned(T), 256, 0, stream>>>(G, dX, dest, topk, gates, scores, logits, dg, centroids,
                                                          centroid_f32, T, d, N, K, du, dz_row, dz_out);
    return cudaGetLastError();
}

cudaError_t launch_centroid_grad(const uint16_t* u, const int32_t* offsets, const int32_t* perm_token,
                                 const float* dz_row, int N, int d, float* de, cudaStream_t stream) {
    const dim3 grid(unsigned(N), unsigned((d + 255) / 256));
    centroid_grad_kernel<<<grid, 256, 0, stream>>>(u, offsets, perm_token, dz_row, d, de);
    return cudaGetLastError();
}

cudaError_t launch_fp8_transpose(const uint8_t* q, const float* s, int G, int rows, int cols, uint8_t* qt, float* st,
                                 cudaStream_t stream) {
    const dim3 grid(unsigned(cols / 128), unsigned(rows / 128), unsigned(G));
    fp8_transpose_kernel<<<grid, 256, 0, stream>>>(q, s, rows, cols, qt, st);
    return cudaGetLastError();
}

cudaError_t launch_sgd_requant(float* w, const float* grad, int G, int rows, int cols, float lr, uint8_t* q, float* s,
                               uint8_t* qt, float* st, cudaStream_t stream) {
    const dim3 grid(unsigned(cols / 128), unsigned(rows / 128), unsigned(G));
    sgd_requant_kernel<<<grid, 256, 0, stream>>>(w, grad, rows, cols, lr, q, s, qt, st);
    return cudaGetLastError();
}

cudaError_t launch_sgd_f32(float* w, const float* grad, int64_t n, float lr, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    sgd_f32_kernel<<<grid_for(n, 256), 256, 0, stream>>>(w, grad, n, lr);
    return cudaGetLastError();
}

}  // namespace moe
