// FP8 E4M3 quantisation with fine-grained scales (DeepSeek-V3 Technical
// Report, learn.ifs.name summary, paragraph on FP8 scaling): one fp32 scale per
// 1x128 activation tile and per 128x128 weight block; scale = amax / 448
// (1 for an all-zero tile) and q = e4m3(x / scale), both IEEE fp32 divisions,
// conversion with round-to-nearest-even and saturation to +-448. The 1x128
// kernel forms x / scale by reciprocal where that gives the same code
// (e4m3_quotient) and divides elsewhere.
//
// Both kernels stream bf16 in and e4m3 out with 16-byte loads; they are HBM
// bound (3 bytes of traffic per element).
#include "common.cuh"
#include "e4m3.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

// One half-warp per 1x128 tile: lane l of the half holds elements 8l..8l+7.
// Tiles are visited row-major, so a warp reads 512 contiguous bytes.
__global__ void __launch_bounds__(256) quant_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                          int64_t ld_x, uint8_t* __restrict__ q,
                                                          float* __restrict__ scales, int64_t ld_s) {
    const int64_t tiles_per_row = cols / 128;
    const int64_t n_tiles = rows * tiles_per_row;
    const int half = (threadIdx.x & 31) >> 4, l = threadIdx.x & 15;
    const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t warp_stride = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t0 = warp_global * 2; t0 < n_tiles; t0 += warp_stride * 2) {
        const int64_t t = t0 + half;
        const bool active = t < n_tiles;
        const int64_t r = active ? t / tiles_per_row : 0;
        const int64_t kb = active ? t - r * tiles_per_row : 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (active) v = __ldg(reinterpret_cast<const uint4*>(x + r * ld_x + kb * 128) + l);
        float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = tile_scale(amax), rc = e4m3_recip(sc);
        if (active) {
            uint32_t w0 = pack_e4m3x2(e4m3_quotient(f[0], sc, rc), e4m3_quotient(f[1], sc, rc)) |
                          (pack_e4m3x2(e4m3_quotient(f[2], sc, rc), e4m3_quotient(f[3], sc, rc)) << 16);
            uint32_t w1 = pack_e4m3x2(e4m3_quotient(f[4], sc, rc), e4m3_quotient(f[5], sc, rc)) |
                          (pack_e4m3x2(e4m3_quotient(f[6], sc, rc), e4m3_quotient(f[7], sc, rc)) << 16);
            reinterpret_cast<uint2*>(q + r * cols + kb * 128)[l] = make_uint2(w0, w1);
            if (l == 0) scales[kb * ld_s + r] = sc;
        }
    }
}

// One block of 256 threads per 128x128 weight block: thread t covers rows
// t/16 + 16i (i < 8) and columns 8*(t%16) .. +7 of the block.
__global__ void __launch_bounds__(256) quant_128x128_kernel(const uint16_t* __restrict__ w, int64_t rows,
                                                            int64_t cols, uint8_t* __restrict__ q,
                                                            float* __restrict__ scales) {
    __shared__ float warp_max[8];
    const int64_t bc = blockIdx.x, br = blockIdx.y;
    const int t = threadIdx.x;
    const int64_t r0 = br * 128 + t / 16;
    const int64_t c0 = bc * 128 + (t % 16) * 8;
    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + 16 * i;
        v[i] = r < rows ? __ldg(reinterpret_cast<const uint4*>(w + r * cols + c0)) : make_uint4(0, 0, 0, 0);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[i].x)), fabsf(bf16_hi(v[i].x))),
                                 fmaxf(fabsf(bf16_lo(v[i].y)), fabsf(bf16_hi(v[i].y)))));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[i].z)), fabsf(bf16_hi(v[i].z))),
                                 fmaxf(fabsf(bf16_lo(v[i].w)), fabsf(bf16_hi(v[i].w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((t & 31) == 0) warp_max[t >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float sc = tile_scale(amax);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + 16 * i;
        if (r < rows) {
            uint32_t w0 = pack_e4m3x2(__fdiv_rn(bf16_lo(v[i].x), sc), __fdiv_rn(bf16_hi(v[i].x), sc)) |
                          (pack_e4m3x2(__fdiv_rn(bf16_lo(v[i].y), sc), __fdiv_rn(bf16_hi(v[i].y), sc)) << 16);
            uint32_t w1 = pack_e4m3x2(__fdiv_rn(bf16_lo(v[i].z), sc), __fdiv_rn(bf16_hi(v[i].z), sc)) |
                          (pack_e4m3x2(__fdiv_rn(bf16_lo(v[i].w), sc), __fdiv_rn(bf16_hi(v[i].w), sc)) << 16);
            *reinterpret_cast<uint2*>(q + r * cols + c0) = make_uint2(w0, w1);
        }
    }
    if (t == 0) scales[br * (cols / 128) + bc] = sc;
}

}  // namespace

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                               float* scales, int64_t ld_s, cudaStream_t stream) {
    const int64_t n_tiles = rows * (cols / 128);
    if (n_tiles == 0) return cudaSuccess;
    const int64_t warps = (n_tiles + 1) / 2;
    int64_t blocks = (warps + 7) / 8;
    const int64_t cap = int64_t(num_sms()) * 8;   // 8 blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    quant_1x128_kernel<<<int(blocks), 256, 0, stream>>>(x, rows, cols, ld_x, q, scales, ld_s);
    return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, float* scales,
                                 cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    dim3 grid(unsigned(cols / 128), unsigned((rows + 127) / 128));
    quant_128x128_kernel<<<grid, 256, 0, stream>>>(w, rows, cols, q, scales);
    return cudaGetLastError();
}

}  // namespace moe
