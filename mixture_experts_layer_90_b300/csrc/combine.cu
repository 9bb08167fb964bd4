// Combine and bias update.
//
// Combine (nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)", "The
// notation"): h'_t = u_t + y_shared_t + sum_k g_{t,k} y_{dest_row[t,k]},
// accumulated in fp32 in that order, stored as bf16. One warp per (token, 256
// columns), 16-byte loads of every row it reads; HBM bound ((K + 3) rows of
// traffic per token). Small batches (decode) still give every SM work: a warp
// per token walking its columns left 8 SMs busy at T = 64, bound by load latency.
//
// Bias update (learn.ifs.name summary, bias paragraph): after the step an
// overloaded expert's bias falls by gamma and an underloaded one's rises;
// overloaded means load * N > T * K (above the mean), one fp32 addition.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ u, const uint16_t* __restrict__ ys,
                                                      const uint16_t* __restrict__ y, const float* __restrict__ gates,
                                                      const int32_t* __restrict__ dest_row, int64_t T, int d, int K,
                                                      int64_t R, uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int chunks = (d + 255) / 256;
    const int64_t items = T * chunks;
    for (int64_t item = int64_t(blockIdx.x) * 8 + w; item < items; item += int64_t(gridDim.x) * 8) {
        const int64_t t = item / chunks;
        const int c0 = int(item - t * chunks) * 256;
        int my_row = 0;
        float my_g = 0.0f;
        if (lane < K) {
            my_row = __ldg(dest_row + t * K + lane);
            my_g = __ldg(gates + t * K + lane);
            if (my_row < 0 || my_row >= R) {
                report(MOE_ERR_DEVICE_DATA);
                my_row = 0;
                my_g = 0.0f;
            }
        }
        {
            const int c = c0 + lane * 8;
            const bool active = c < d;
            float acc[8];
            uint4 uv = make_uint4(0, 0, 0, 0);
            if (active) uv = __ldg(reinterpret_cast<const uint4*>(u + t * d + c));
            acc[0] = bf16_lo(uv.x); acc[1] = bf16_hi(uv.x); acc[2] = bf16_lo(uv.y); acc[3] = bf16_hi(uv.y);
            acc[4] = bf16_lo(uv.z); acc[5] = bf16_hi(uv.z); acc[6] = bf16_lo(uv.w); acc[7] = bf16_hi(uv.w);
            if (ys && active) {
                const uint4 sv = __ldg(reinterpret_cast<const uint4*>(ys + t * d + c));
                acc[0] += bf16_lo(sv.x); acc[1] += bf16_hi(sv.x); acc[2] += bf16_lo(sv.y); acc[3] += bf16_hi(sv.y);
                acc[4] += bf16_lo(sv.z); acc[5] += bf16_hi(sv.z); acc[6] += bf16_lo(sv.w); acc[7] += bf16_hi(sv.w);
            }
            for (int k = 0; k < K; ++k) {
                const int row = __shfl_sync(0xffffffffu, my_row, k);
                const float g = __shfl_sync(0xffffffffu, my_g, k);
                if (!active) continue;
                const uint4 yv = __ldg(reinterpret_cast<const uint4*>(y + int64_t(row) * d + c));
                acc[0] = fmaf(g, bf16_lo(yv.x), acc[0]); acc[1] = fmaf(g, bf16_hi(yv.x), acc[1]);
                acc[2] = fmaf(g, bf16_lo(yv.y), acc[2]); acc[3] = fmaf(g, bf16_hi(yv.y), acc[3]);
                acc[4] = fmaf(g, bf16_lo(yv.z), acc[4]); acc[5] = fmaf(g, bf16_hi(yv.z), acc[5]);
                acc[6] = fmaf(g, bf16_lo(yv.w), acc[6]); acc[7] = fmaf(g, bf16_hi(yv.w), acc[7]);
            }
            if (active)
                *reinterpret_cast<uint4*>(out + t * d + c) =
                    make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                               pack_bf16x2(acc[6], acc[7]));
        }
    }
}

__global__ void bias_update_kernel(float* __restrict__ bias, const int32_t* __restrict__ loads, int N, int64_t T,
                                   int K, float gamma) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    const int64_t lhs = int64_t(loads[i]) * N, mean_num = T * K;
    if (lhs > mean_num) bias[i] = __fsub_rn(bias[i], gamma);
    else if (lhs < mean_num) bias[i] = __fadd_rn(bias[i], gamma);
}

// One thread waits on an mbarrier that nothing arrives on, with the same
// bounded wait as the pipelines (a limit of `limit_ns`): it must give up,
// record MOE_ERR_TIMEOUT in the status word and return.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    mbar_wait_for(smem_u32(&bar), 0, &abort_flag, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y_perm, const float* gates,
                           const int32_t* dest_row, int64_t T, int d, int K, int64_t R, uint16_t* out,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    int64_t blocks = (T * ((d + 255) / 256) + 7) / 8;   // a warp per (token, 256 columns)
    const int64_t cap = int64_t(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    combine_kernel<<<int(blocks), 256, 0, stream>>>(u, y_shared, y_perm, gates, dest_row, T, d, K, R, out);
    return cudaGetLastError();
}

cudaError_t launch_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma,
                               cudaStream_t stream) {
    bias_update_kernel<<<(N + 255) / 256, 256, 0, stream>>>(bias, loads, N, T, K, gamma);
    return cudaGetLastError();
}

}  // namespace moe
