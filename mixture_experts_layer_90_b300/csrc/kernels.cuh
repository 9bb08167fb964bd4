// Launchers of the memory-bound kernels (quant.cu, route.cu, permute.cu,
// combine.cu). Arguments are validated by the C ABI layer (abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

int num_sms();

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                               float* scales, int64_t ld_s, cudaStream_t stream);
cudaError_t launch_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, float* scales,
                                 cudaStream_t stream);

// Routing: bf16 split of the centroids (prepared once per set of centroids),
// tensor-core gate logits, selection.
struct RoutePlan {
    int terms;      // 3 for fp32 centroids (exact bf16 split), 1 for bf16
    int n_pad;      // N rounded up to 256
    int splits;     // split-K parts of the gate GEMM
    size_t split_bytes, zpart_bytes, total_bytes;
};
size_t prepared_centroid_bytes(int d, int N, int centroid_dtype);
RoutePlan plan_route(int64_t T, int d, int N, int centroid_dtype);
cudaError_t launch_route_prepare(const void* centroids, int centroid_dtype, int N, int d, const RoutePlan& plan,
                                 void* prepared, cudaStream_t stream);
cudaError_t launch_route(const uint16_t* u, int64_t T, int d, const void* prepared, const float* bias, int N, int K,
                         int n_groups, int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                         float* scores, void* zpart_ws, const RoutePlan& plan, cudaStream_t stream);

// Permutation (stable counting sort by expert) and row scatter.
size_t permute_ws_bytes(int64_t T, int N);
cudaError_t launch_permute(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K, int out_dtype,
                           int with_shared, int32_t* offsets, int32_t* perm_token, int32_t* dest_row, void* x_perm,
                           float* x_perm_scales, void* ws, cudaStream_t stream);

// Sequence-wise balance statistics (balance.cu).
size_t balance_ws_bytes(int64_t T, int N, int64_t seq_len);
cudaError_t launch_balance(const float* scores, const int32_t* topk_idx, int64_t T, int N, int K, int64_t seq_len,
                           int32_t* seq_loads, float* seq_prob, float* seq_stat, void* ws, cudaStream_t stream);

cudaError_t launch_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y_perm, const float* gates,
                           const int32_t* dest_row, int64_t T, int d, int K, int64_t R, uint16_t* out,
                           cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma,
                               cudaStream_t stream);

}  // namespace moe
