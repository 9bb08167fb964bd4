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
// logits (optional): the fp32 gate logits z [T, N] (the training forward keeps them)
cudaError_t launch_route(const uint16_t* u, int64_t T, int d, const void* prepared, const float* bias, int N, int K,
                         int n_groups, int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                         float* scores, void* zpart_ws, const RoutePlan& plan, cudaStream_t stream,
                         float* logits = nullptr);

// Permutation (stable counting sort by expert) and row scatter.
size_t permute_ws_bytes(int64_t T, int N);
cudaError_t launch_permute(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K, int out_dtype,
                           int with_shared, int32_t* offsets, int32_t* perm_token, int32_t* dest_row, void* x_perm,
                           float* x_perm_scales, void* ws, cudaStream_t stream, int32_t* loads = nullptr);

// Sequence-wise balance statistics (balance.cu).
size_t balance_ws_bytes(int64_t T, int N, int64_t seq_len);
cudaError_t launch_balance(const float* scores, const int32_t* topk_idx, int64_t T, int N, int K, int64_t seq_len,
                           int32_t* seq_loads, float* seq_prob, float* seq_stat, void* ws, cudaStream_t stream);

cudaError_t launch_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y_perm, const float* gates,
                           const int32_t* dest_row, int64_t T, int d, int K, int64_t R, uint16_t* out,
                           cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);

// Backward pass and training step (backward.cu).
enum { kQuantTScaledG = 0, kQuantTTokens = 1, kQuantTRows = 2, kQuantTSwiglu = 3 };
cudaError_t launch_combine_bwd(const uint16_t* G, const uint16_t* y, const float* gates, const int32_t* dest,
                               int64_t T, int d, int K, int64_t R, uint8_t* qdy, float* sdy, float* row_gate,
                               float* dg, cudaStream_t stream);
cudaError_t launch_swiglu_bwd(const uint16_t* dA, const uint16_t* H, int64_t R, int I, uint16_t* dH, uint8_t* qdh,
                              float* sdh, cudaStream_t stream);
cudaError_t launch_kblock_offsets(const int32_t* offsets, int G, int32_t* kofs, cudaStream_t stream);
cudaError_t launch_pad_rows(const int32_t* offsets, const int32_t* kofs, int G, int64_t Kp, int32_t* prow,
                            cudaStream_t stream);
cudaError_t launch_quant_t(int src_kind, const int32_t* prow, const int32_t* kofs, int G, int64_t TK,
                           const int32_t* perm_token, const float* row_gate, const uint16_t* src, int C,
                           int64_t Kp, uint8_t* q, float* s, cudaStream_t stream);
cudaError_t launch_unpermute_bwd(const uint16_t* G, const uint16_t* dX, const int32_t* dest, const int32_t* topk,
                                 const float* gates, const float* scores, const float* logits, const float* dg,
                                 const void* centroids,
                                 int centroid_f32, int64_t T, int d, int N, int K, uint16_t* du, float* dz_row,
                                 float* dz_out, cudaStream_t stream);
cudaError_t launch_centroid_grad(const uint16_t* u, const int32_t* offsets, const int32_t* perm_token,
                                 const float* dz_row, int N, int d, float* de, cudaStream_t stream);
cudaError_t launch_fp8_transpose(const uint8_t* q, const float* s, int G, int rows, int cols, uint8_t* qt, float* st,
                                 cudaStream_t stream);
cudaError_t launch_sgd_requant(float* w, const float* grad, int G, int rows, int cols, float lr, uint8_t* q, float* s,
                               uint8_t* qt, float* st, cudaStream_t stream);
cudaError_t launch_sgd_f32(float* w, const float* grad, int64_t n, float lr, cudaStream_t stream);
cudaError_t launch_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma,
                               cudaStream_t stream);

}  // namespace moe
