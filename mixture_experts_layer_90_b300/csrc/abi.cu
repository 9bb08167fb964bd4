// The C ABI (include/moe.h): argument validation, workspace layout and the
// launch sequence of the layer. No entry point allocates device memory.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

namespace moe {


int num_sms() {
    // SM count of the current device, looked up once per device
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace moe

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
bool al32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
size_t up256(size_t x) { return (x + 255) / 256 * 256; }

#define REQUIRE(cond, ...)                                    \
    do {                                                      \
        if (!(cond)) return fail(MOE_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)
#define UNSUPPORTED(cond, ...)                                \
    do {                                                      \
        if (!(cond)) return fail(MOE_ERR_UNSUPPORTED, __VA_ARGS__); \
    } while (0)
#define CUDA_OK(expr)                                                                              \
    do {                                                                                           \
        cudaError_t e_ = (expr);                                                                   \
        if (e_ != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
    } while (0)
#define STATUS_OK(expr)                  \
    do {                                 \
        moe_status s_ = (expr);          \
        if (s_ != MOE_OK) return s_;     \
    } while (0)

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

moe_status check_route(const uint16_t* u, int64_t T, int d, const void* centroids, int cdt, const float* bias, int N,
                       int K, int n_groups, int topk_groups, const int32_t* idx, const float* gates,
                       const int32_t* loads) {
    REQUIRE(T >= 0 && T <= kMaxRows, "moe_route: T=%lld out of range", (long long)T);
    REQUIRE(d > 0 && d % 64 == 0, "moe_route: d=%d must be a positive multiple of 64", d);
    REQUIRE(K >= 1 && K <= 16 && K <= N, "moe_route: K=%d must satisfy 1 <= K <= min(16, N)", K);
    REQUIRE(N >= 1 && N <= 1024, "moe_route: N=%d must be in [1, 1024]", N);
    REQUIRE(cdt == MOE_DTYPE_F32 || cdt == MOE_DTYPE_BF16, "moe_route: centroid dtype %d", cdt);
    REQUIRE(n_groups >= 1 && n_groups <= 32 && N % n_groups == 0, "moe_route: n_groups=%d must divide N", n_groups);
    if (n_groups > 1) {
        REQUIRE(N / n_groups >= 2, "moe_route: groups need at least two experts");
        REQUIRE(topk_groups >= 1 && topk_groups <= n_groups, "moe_route: topk_groups=%d", topk_groups);
        REQUIRE(topk_groups * (N / n_groups) >= K, "moe_route: kept groups hold fewer than K experts");
    }
    if (T == 0) return MOE_OK;   // no token: only the loads are written (zero)
    REQUIRE(u && centroids && bias && idx && gates, "moe_route: null pointer");
    REQUIRE(al16(u) && al16(centroids), "moe_route: u and centroids must be 16-byte aligned");
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err; }

int moe_num_sms(void) { return moe::num_sms(); }

moe_status moe_get_device_status(moe_stream_t stream, int* status) {
    REQUIRE(status, "moe_get_device_status: null status");
    CUDA_OK(cudaStreamSynchronize(stream));
    int v = 0, zero = 0;
    CUDA_OK(cudaMemcpyFromSymbol(&v, moe::g_device_status, sizeof(int)));
    CUDA_OK(cudaMemcpyToSymbol(moe::g_device_status, &zero, sizeof(int)));
    *status = v;
    return MOE_OK;
}

moe_status fp8_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q, float* scales,
                           int64_t ld_s, moe_stream_t stream) {
    REQUIRE(rows >= 0 && cols > 0 && cols % 128 == 0, "fp8_quant_1x128: cols=%lld must be a multiple of 128",
            (long long)cols);
    REQUIRE(ld_x >= cols && ld_x % 8 == 0, "fp8_quant_1x128: ld_x must be >= cols and a multiple of 8");
    REQUIRE(ld_s >= rows, "fp8_quant_1x128: ld_s must be >= rows");
    if (rows == 0) return MOE_OK;
    REQUIRE(x && q && scales, "fp8_quant_1x128: null pointer");
    REQUIRE(al16(x) && al8(q), "fp8_quant_1x128: x must be 16-byte and q 8-byte aligned");
    CUDA_OK(moe::launch_quant_1x128(x, rows, cols, ld_x, q, scales, ld_s, stream));
    return MOE_OK;
}

moe_status fp8_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, float* scales,
                             moe_stream_t stream) {
    REQUIRE(rows >= 0 && cols > 0 && cols % 128 == 0, "fp8_quant_128x128: cols must be a multiple of 128");
    REQUIRE((rows + 127) / 128 <= 65535 && cols / 128 <= int64_t(1) << 30, "fp8_quant_128x128: too many blocks");
    if (rows == 0) return MOE_OK;
    REQUIRE(w && q && scales, "fp8_quant_128x128: null pointer");
    REQUIRE(al16(w) && al8(q), "fp8_quant_128x128: w must be 16-byte and q 8-byte aligned");
    CUDA_OK(moe::launch_quant_128x128(w, rows, cols, q, scales, stream));
    return MOE_OK;
}

size_t moe_route_workspace_size(int64_t T, int d, int N, int centroid_dtype) {
    return moe::plan_route(T, d, N, centroid_dtype).total_bytes;
}

size_t moe_route_prepared_centroids_size(int d, int N, int centroid_dtype) {
    return moe::prepared_centroid_bytes(d, N, centroid_dtype);
}

size_t moe_route_prepared_workspace_size(int64_t T, int d, int N, int centroid_dtype) {
    return moe::plan_route(T, d, N, centroid_dtype).zpart_bytes;
}

moe_status moe_route_prepare_centroids(const void* centroids, int centroid_dtype, int N, int d, void* prepared,
                                       size_t prepared_bytes, moe_stream_t stream) {
    REQUIRE(d > 0 && d % 64 == 0, "moe_route_prepare_centroids: d=%d must be a positive multiple of 64", d);
    REQUIRE(N >= 1 && N <= 1024, "moe_route_prepare_centroids: N=%d must be in [1, 1024]", N);
    REQUIRE(centroid_dtype == MOE_DTYPE_F32 || centroid_dtype == MOE_DTYPE_BF16,
            "moe_route_prepare_centroids: centroid dtype %d", centroid_dtype);
    REQUIRE(centroids && prepared, "moe_route_prepare_centroids: null pointer");
    const moe::RoutePlan plan = moe::plan_route(0, d, N, centroid_dtype);
    if (prepared_bytes < plan.split_bytes || (reinterpret_cast<uintptr_t>(prepared) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_route_prepare_centroids: needs %zu bytes, 256-byte aligned",
                    plan.split_bytes);
    CUDA_OK(moe::launch_route_prepare(centroids, centroid_dtype, N, d, plan, prepared, stream));
    return MOE_OK;
}

// logits (optional, the training forward's): the fp32 gate logits [T, N]
static moe_status route_prepared_impl(const uint16_t* u, int64_t T, int d, const void* prepared, int centroid_dtype,
                                      const float* bias, int N, int K, int n_groups, int topk_groups,
                                      int32_t* topk_idx, float* gates, int32_t* loads, float* scores,
                                      void* workspace, size_t workspace_bytes, moe_stream_t stream, float* logits) {
    STATUS_OK(check_route(u, T, d, prepared, centroid_dtype, bias, N, K, n_groups, topk_groups, topk_idx, gates,
                          loads));
    const moe::RoutePlan plan = moe::plan_route(T, d, N, centroid_dtype);
    if (T > 0 && (reinterpret_cast<uintptr_t>(prepared) & 255u))
        return fail(MOE_ERR_INVALID_ARG, "moe_route_prepared: prepared centroids must be 256-byte aligned");
    if (T > 0 && (!workspace || workspace_bytes < plan.zpart_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(MOE_ERR_WORKSPACE, "moe_route_prepared: workspace needs %zu bytes, 256-byte aligned",
                    plan.zpart_bytes);
    CUDA_OK(moe::launch_route(u, T, d, prepared, bias, N, K, n_groups > 1 ? n_groups : 1,
                              n_groups > 1 ? topk_groups : 1, topk_idx, gates, loads, scores, workspace, plan, stream,
                              logits));
    return MOE_OK;
}

moe_status moe_route_prepared(const uint16_t* u, int64_t T, int d, const void* prepared, int centroid_dtype,
                              const float* bias, int N, int K, int n_groups, int topk_groups, int32_t* topk_idx,
                              float* gates, int32_t* loads, float* scores, void* workspace, size_t workspace_bytes,
                              moe_stream_t stream) {
    REQUIRE(loads, "moe_route: null loads");
    return route_prepared_impl(u, T, d, prepared, centroid_dtype, bias, N, K, n_groups, topk_groups, topk_idx, gates,
                               loads, scores, workspace, workspace_bytes, stream, nullptr);
}

static moe_status route_impl(const uint16_t* u, int64_t T, int d, const void* centroids, int centroid_dtype,
                             const float* bias, int N, int K, int n_groups, int topk_groups, int32_t* topk_idx,
                             float* gates, int32_t* loads, float* scores, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream, float* logits) {
    STATUS_OK(check_route(u, T, d, centroids, centroid_dtype, bias, N, K, n_groups, topk_groups, topk_idx, gates,
                          loads));
    const moe::RoutePlan plan = moe::plan_route(T, d, N, centroid_dtype);
    if (!workspace || workspace_bytes < plan.total_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_route: workspace needs %zu bytes, 256-byte aligned", plan.total_bytes);
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    if (T > 0) CUDA_OK(moe::launch_route_prepare(centroids, centroid_dtype, N, d, plan, ws, stream));
    CUDA_OK(moe::launch_route(u, T, d, ws, bias, N, K, n_groups > 1 ? n_groups : 1, n_groups > 1 ? topk_groups : 1,
                              topk_idx, gates, loads, scores, ws + plan.split_bytes, plan, stream, logits));
    return MOE_OK;
}

moe_status moe_route(const uint16_t* u, int64_t T, int d, const void* centroids, int centroid_dtype, const float* bias,
                     int N, int K, int n_groups, int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                     float* scores, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    REQUIRE(loads, "moe_route: null loads");
    return route_impl(u, T, d, centroids, centroid_dtype, bias, N, K, n_groups, topk_groups, topk_idx, gates, loads,
                      scores, workspace, workspace_bytes, stream, nullptr);
}

size_t moe_route_balance_stats_workspace_size(int64_t T, int N, int64_t seq_len) {
    return moe::balance_ws_bytes(T, N, seq_len);
}

moe_status moe_route_balance_stats(const float* scores, const int32_t* topk_idx, int64_t T, int N, int K,
                                   int64_t seq_len, int32_t* seq_loads, float* seq_prob, float* seq_stat,
                                   void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    REQUIRE(T >= 0 && T <= kMaxRows, "moe_route_balance_stats: T=%lld out of range", (long long)T);
    REQUIRE(N >= 1 && N <= 1024, "moe_route_balance_stats: N=%d must be in [1, 1024]", N);
    REQUIRE(K >= 1 && K <= 16 && K <= N, "moe_route_balance_stats: K=%d", K);
    REQUIRE(seq_len >= 1, "moe_route_balance_stats: seq_len=%lld must be positive", (long long)seq_len);
    if (T == 0) return MOE_OK;
    REQUIRE((T + seq_len - 1) / seq_len <= 0x7fffffff, "moe_route_balance_stats: too many sequences");
    REQUIRE(scores && topk_idx && seq_loads && seq_prob && seq_stat, "moe_route_balance_stats: null pointer");
    const size_t need = moe::balance_ws_bytes(T, N, seq_len);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return fail(MOE_ERR_WORKSPACE, "moe_route_balance_stats: workspace needs %zu bytes", need);
    CUDA_OK(moe::launch_balance(scores, topk_idx, T, N, K, seq_len, seq_loads, seq_prob, seq_stat, workspace,
                                stream));
    return MOE_OK;
}

size_t moe_permute_workspace_size(int64_t T, int N) { return moe::permute_ws_bytes(T, N); }

// loads (internal, may be null): the per-expert pair counts, written by the permutation
// (the layer takes its loads from here instead of from the routing)
static moe_status permute_impl(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K,
                               int out_dtype, int with_shared, int32_t* offsets, int32_t* perm_token, int32_t* dest_row,
                               void* x_perm, float* x_perm_scales, void* workspace, size_t workspace_bytes,
                               moe_stream_t stream, int32_t* loads) {
    REQUIRE(T >= 0 && T * (K + 1) <= kMaxRows, "moe_permute: T=%lld out of range", (long long)T);
    REQUIRE(d > 0 && d % 128 == 0, "moe_permute: d=%d must be a multiple of 128", d);
    REQUIRE(N >= 1 && N <= 1024, "moe_permute: N=%d must be in [1, 1024]", N);
    REQUIRE(K >= 1 && K <= 16 && K <= N, "moe_permute: K=%d", K);
    REQUIRE(out_dtype == MOE_DTYPE_BF16 || out_dtype == MOE_DTYPE_E4M3, "moe_permute: out dtype %d", out_dtype);
    REQUIRE(offsets, "moe_permute: null offsets");
    if (T > 0) {
        REQUIRE(x && topk_idx && perm_token && dest_row && x_perm, "moe_permute: null pointer");
        REQUIRE(out_dtype != MOE_DTYPE_E4M3 || x_perm_scales, "moe_permute: E4M3 output needs scales");
        REQUIRE(al16(x) && al16(x_perm), "moe_permute: x and x_perm must be 16-byte aligned");
    }
    const size_t need = moe::permute_ws_bytes(T, N);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return fail(MOE_ERR_WORKSPACE, "moe_permute: workspace needs %zu bytes", need);
    CUDA_OK(moe::launch_permute(x, T, d, topk_idx, N, K, out_dtype, with_shared ? 1 : 0, offsets, perm_token,
                                dest_row, x_perm, x_perm_scales, workspace, stream, loads));
    return MOE_OK;
}

moe_status moe_permute(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K, int out_dtype,
                       int with_shared, int32_t* offsets, int32_t* perm_token, int32_t* dest_row, void* x_perm,
                       float* x_perm_scales, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return permute_impl(x, T, d, topk_idx, N, K, out_dtype, with_shared, offsets, perm_token, dest_row, x_perm,
                        x_perm_scales, workspace, workspace_bytes, stream, nullptr);
}

// fp8_grouped_gemm; with h_out (MOE_EPI_SWIGLU_FP8 only) the products are also
// stored in bf16 [M_total, Nd] (the training forward keeps them). With a_gather,
// A is [a_rows][Kd] and the grouped A's row r is its row a_gather[r] (r < tk) or
// r - tk; sa is [Kd/128][a_rows].
static moe_status fp8_gemm_impl(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                                const int32_t* group_offsets, int G, int64_t M_total, int Nd, int Kd, int epilogue,
                                void* C, float* c_scales, uint16_t* h_out, moe_stream_t stream,
                                const int32_t* a_gather = nullptr, int64_t tk = 0, int64_t a_rows = 0) {
    REQUIRE(G >= 1 && G <= moe::gemm_max_groups(), "fp8_grouped_gemm: G=%d must be in [1, 1024]", G);
    REQUIRE(M_total >= 0 && M_total <= kMaxRows, "fp8_grouped_gemm: M_total out of range");
    REQUIRE(Kd > 0 && Kd % 128 == 0, "fp8_grouped_gemm: Kd=%d must be a multiple of 128", Kd);
    REQUIRE(Nd > 0 && Nd % 256 == 0, "fp8_grouped_gemm: Nd=%d must be a multiple of 256", Nd);
    REQUIRE(int64_t(G) * Nd <= kMaxRows, "fp8_grouped_gemm: G*Nd too large");
    REQUIRE(epilogue == MOE_EPI_BF16 || epilogue == MOE_EPI_SWIGLU_FP8, "fp8_grouped_gemm: epilogue %d", epilogue);
    REQUIRE(group_offsets && B && sb, "fp8_grouped_gemm: null pointer");
    REQUIRE(al16(B), "fp8_grouped_gemm: B must be 16-byte aligned");
    if (M_total == 0) return MOE_OK;
    REQUIRE(A && sa && C, "fp8_grouped_gemm: null pointer");
    REQUIRE(epilogue != MOE_EPI_SWIGLU_FP8 || c_scales, "fp8_grouped_gemm: SwiGLU output needs scales");
    REQUIRE(al16(A) && al32(C), "fp8_grouped_gemm: A must be 16-byte and C 32-byte aligned");
    REQUIRE(!a_gather || (a_rows > 0 && tk >= 0 && tk <= M_total), "fp8_grouped_gemm: bad row gather");
    CUtensorMap ta, tb;
    if (!moe::make_kmajor_map(&ta, A, false, uint64_t(Kd), uint64_t(a_gather ? a_rows : M_total), uint64_t(Kd), 128) ||
        !moe::make_kmajor_map(&tb, B, false, uint64_t(Kd), uint64_t(G) * Nd, uint64_t(Kd), 256))
        return fail(MOE_ERR_CUDA, "fp8_grouped_gemm: tensor map encoding failed");
    moe::GemmArgs a{};
    a.group_offsets = group_offsets;
    a.G = G;
    a.M_total = M_total;
    a.Nd = Nd;
    a.Kd = Kd;
    a.k_steps = Kd / 128;
    a.a_k_repeat = 1;
    a.elems_per_step = 128;
    a.splits = 1;
    a.epilogue = epilogue;
    a.sa = sa;
    a.lda_s = a_gather ? a_rows : M_total;
    a.sb = sb;
    a.C = C;
    a.c_scales = c_scales;
    a.h_out = h_out;
    a.a_gather = a_gather;
    a.a_gather_tk = tk;
    a.a_src = A;
    REQUIRE(!h_out || (epilogue == MOE_EPI_SWIGLU_FP8 && al32(h_out)), "fp8_grouped_gemm: bad product output");
    CUDA_OK(moe::run_grouped_gemm(moe::kModeFP8, ta, tb, a, moe::num_sms(), stream));
    return MOE_OK;
}

moe_status fp8_grouped_gemm(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                            const int32_t* group_offsets, int G, int64_t M_total, int Nd, int Kd, int epilogue,
                            void* C, float* c_scales, moe_stream_t stream) {
    return fp8_gemm_impl(A, sa, B, sb, group_offsets, G, M_total, Nd, Kd, epilogue, C, c_scales, nullptr, stream);
}

moe_status bf16_grouped_gemm(const uint16_t* A, const uint16_t* B, const int32_t* group_offsets, int G,
                             int64_t M_total, int Nd, int Kd, int epilogue, void* C, moe_stream_t stream) {
    REQUIRE(G >= 1 && G <= moe::gemm_max_groups(), "bf16_grouped_gemm: G=%d must be in [1, 1024]", G);
    REQUIRE(M_total >= 0 && M_total <= kMaxRows, "bf16_grouped_gemm: M_total out of range");
    REQUIRE(Kd > 0 && Kd % 64 == 0, "bf16_grouped_gemm: Kd=%d must be a multiple of 64", Kd);
    REQUIRE(Nd > 0 && Nd % 256 == 0, "bf16_grouped_gemm: Nd=%d must be a multiple of 256", Nd);
    REQUIRE(int64_t(G) * Nd <= kMaxRows, "bf16_grouped_gemm: G*Nd too large");
    REQUIRE(epilogue == MOE_EPI_BF16 || epilogue == MOE_EPI_SWIGLU_BF16 || epilogue == MOE_EPI_F32,
            "bf16_grouped_gemm: epilogue %d", epilogue);
    REQUIRE(group_offsets && B, "bf16_grouped_gemm: null pointer");
    REQUIRE(al16(B), "bf16_grouped_gemm: B must be 16-byte aligned");
    if (M_total == 0) return MOE_OK;
    REQUIRE(A && C, "bf16_grouped_gemm: null pointer");
    REQUIRE(al16(A) && al32(C), "bf16_grouped_gemm: A must be 16-byte and C 32-byte aligned");
    CUtensorMap ta, tb;
    if (!moe::make_kmajor_map(&ta, A, true, uint64_t(Kd), uint64_t(M_total), uint64_t(Kd) * 2, 128) ||
        !moe::make_kmajor_map(&tb, B, true, uint64_t(Kd), uint64_t(G) * Nd, uint64_t(Kd) * 2, 256))
        return fail(MOE_ERR_CUDA, "bf16_grouped_gemm: tensor map encoding failed");
    moe::GemmArgs a{};
    a.group_offsets = group_offsets;
    a.G = G;
    a.M_total = M_total;
    a.Nd = Nd;
    a.Kd = Kd;
    a.k_steps = Kd / 64;
    a.a_k_repeat = 1;
    a.elems_per_step = 64;
    a.splits = 1;
    a.promote_steps = moe::kBf16PromoteSteps;
    a.epilogue = epilogue;
    a.C = C;
    CUDA_OK(moe::run_grouped_gemm(moe::kModeBF16, ta, tb, a, moe::num_sms(), stream));
    return MOE_OK;
}

moe_status moe_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y_perm, const float* gates,
                       const int32_t* dest_row, int64_t T, int d, int K, int64_t R, uint16_t* out,
                       moe_stream_t stream) {
    REQUIRE(T >= 0 && d > 0 && d % 8 == 0, "moe_combine: d=%d must be a multiple of 8", d);
    REQUIRE(K >= 1 && K <= 16, "moe_combine: K=%d", K);
    if (T == 0) return MOE_OK;
    REQUIRE(u && y_perm && gates && dest_row && out, "moe_combine: null pointer");
    REQUIRE(al16(u) && al16(y_perm) && al16(out) && (!y_shared || al16(y_shared)),
            "moe_combine: row pointers must be 16-byte aligned");
    CUDA_OK(moe::launch_combine(u, y_shared, y_perm, gates, dest_row, T, d, K, R, out, stream));
    return MOE_OK;
}

moe_status moe_selftest_wait_timeout(int64_t limit_ns, moe_stream_t stream) {
    REQUIRE(limit_ns > 0 && limit_ns <= 1000000000, "moe_selftest_wait_timeout: limit %lld ns not in (0, 1 s]",
            (long long)limit_ns);
    CUDA_OK(moe::launch_wait_timeout_selftest(uint64_t(limit_ns), stream));
    return MOE_OK;
}

moe_status moe_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma,
                           moe_stream_t stream) {
    REQUIRE(N >= 1 && T >= 0 && K >= 1, "moe_bias_update: bad sizes");
    REQUIRE(bias && loads, "moe_bias_update: null pointer");
    CUDA_OK(moe::launch_bias_update(bias, loads, N, T, K, gamma, stream));
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// The layer
// ---------------------------------------------------------------------------

namespace {

struct LayerWs {
    size_t route, perm, offsets, perm_token, dest_row, topk, gates, x_perm, x_scales, act, act_scales, y, u_dev,
        out_dev, total;
};

// host_slots: device copies of u and h' kept in the workspace (0: none; 1: the
// host-buffer call; 2: the pipelined host-buffer call, slots alternating)
LayerWs layer_ws(const moe_layer_weights* w, int64_t T, int host_slots) {
    LayerWs L{};
    const int64_t R = T * w->K + T;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += up256(bytes);
        return at;
    };
    const moe::RoutePlan rp = moe::plan_route(T, w->d, w->N, w->centroid_dtype);
    L.route = take(w->centroids_prepared ? rp.zpart_bytes : rp.total_bytes);
    L.perm = take(moe::permute_ws_bytes(T, w->N));
    L.offsets = take(size_t(w->N + 2) * 4);
    L.perm_token = take(size_t(T) * w->K * 4);
    L.dest_row = take(size_t(T) * w->K * 4);
    L.topk = take(size_t(T) * w->K * 4);
    L.gates = take(size_t(T) * w->K * 4);
    const size_t es = w->fp8 ? 1 : 2;
    L.x_perm = take(size_t(R) * w->d * es);
    L.x_scales = take(w->fp8 ? size_t(w->d / 128) * R * 4 : 0);
    L.act = take(size_t(R) * w->I * es);
    L.act_scales = take(w->fp8 ? size_t(w->I / 128) * R * 4 : 0);
    L.y = take(size_t(R) * w->d * 2);
    L.u_dev = take(size_t(host_slots) * size_t(T) * w->d * 2);
    L.out_dev = take(size_t(host_slots) * size_t(T) * w->d * 2);
    L.total = o;
    return L;
}

moe_status check_layer(const moe_layer_weights* w) {
    REQUIRE(w, "moe_layer: null weights");
    REQUIRE(w->d > 0 && w->d % 256 == 0, "moe_layer: d=%d must be a multiple of 256", w->d);
    REQUIRE(w->I > 0 && w->I % 128 == 0, "moe_layer: I=%d must be a multiple of 128", w->I);
    REQUIRE(w->N + 1 <= moe::gemm_max_groups(), "moe_layer: too many experts");
    REQUIRE(w->w13 && w->w2 && w->centroids && w->bias, "moe_layer: null weight pointer");
    REQUIRE(!w->fp8 || (w->w13_scales && w->w2_scales), "moe_layer: FP8 weights need scales");
    REQUIRE(w->dispatch == MOE_DISPATCH_SCATTER || w->dispatch == MOE_DISPATCH_GATHER,
            "moe_layer: dispatch=%d", w->dispatch);
    return MOE_OK;
}

}  // namespace

size_t moe_layer_workspace_size(const moe_layer_weights* w, int64_t T) { return w ? layer_ws(w, T, 0).total : 0; }
size_t moe_layer_host_workspace_size(const moe_layer_weights* w, int64_t T) {
    return w ? layer_ws(w, T, 1).total : 0;
}

// scores / logits / h_out (training forward, FP8 only): the affinities and the gate
// logits [T, N] and GEMM 1's products in bf16 [R, 2I] are kept there.
static moe_status layer_forward(const moe_layer_weights* w, const uint16_t* u, int64_t T, uint16_t* out,
                                const moe_layer_outputs* outs, int update_bias, uint8_t* ws, const LayerWs& L,
                                moe_stream_t stream, float* scores = nullptr, uint16_t* h_out = nullptr,
                                float* logits = nullptr) {
    const int K = w->K, N = w->N, d = w->d, I = w->I;
    const int64_t R = T * K + T;
    if (T == 0) {
        // no tokens: every load is 0, equal to the mean, so the bias stays as it is
        CUDA_OK(cudaMemsetAsync(outs->loads, 0, sizeof(int32_t) * N, stream));
        if (outs->stage_events)
            for (int i = 0; i <= MOE_LAYER_STAGES; ++i)
                CUDA_OK(cudaEventRecord(reinterpret_cast<cudaEvent_t>(outs->stage_events[i]), stream));
        return MOE_OK;
    }
    int32_t* topk = outs && outs->topk_idx ? outs->topk_idx : reinterpret_cast<int32_t*>(ws + L.topk);
    float* gates = outs && outs->gates ? outs->gates : reinterpret_cast<float*>(ws + L.gates);
    int32_t* loads = outs->loads;
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    int32_t* dest = reinterpret_cast<int32_t*>(ws + L.dest_row);
    void* const* ev = outs ? outs->stage_events : nullptr;
    auto mark = [&](int i) -> moe_status {
        if (ev) CUDA_OK(cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), stream));
        return MOE_OK;
    };
    STATUS_OK(mark(0));
    // the routing leaves the loads to the permutation, which counts the pairs per expert anyway
    if (w->centroids_prepared)
        STATUS_OK(route_prepared_impl(u, T, d, w->centroids_prepared, w->centroid_dtype, w->bias, N, K, w->n_groups,
                                      w->topk_groups, topk, gates, nullptr, scores, ws + L.route, L.perm - L.route,
                                      stream, logits));
    else
        STATUS_OK(route_impl(u, T, d, w->centroids, w->centroid_dtype, w->bias, N, K, w->n_groups, w->topk_groups,
                             topk, gates, nullptr, scores, ws + L.route, L.perm - L.route, stream, logits));
    STATUS_OK(mark(1));
    int32_t* perm_token = reinterpret_cast<int32_t*>(ws + L.perm_token);
    const bool gather = w->fp8 && w->dispatch == MOE_DISPATCH_GATHER;
    if (gather) {
        // fused dispatch: the tokens quantised once into x_perm's space ([T][d] codes,
        // [d/128][T] scales), the permutation without moving rows; GEMM 1 gathers them
        CUDA_OK(moe::launch_quant_1x128(u, T, d, d, ws + L.x_perm, reinterpret_cast<float*>(ws + L.x_scales), T,
                                        stream));
        CUDA_OK(moe::launch_permute(u, T, d, topk, N, K, MOE_DTYPE_E4M3, 1, offsets, perm_token, dest, nullptr,
                                    nullptr, ws + L.perm, stream, loads));
    } else {
        STATUS_OK(permute_impl(u, T, d, topk, N, K, w->fp8 ? MOE_DTYPE_E4M3 : MOE_DTYPE_BF16, 1, offsets,
                               perm_token, dest, ws + L.x_perm, reinterpret_cast<float*>(ws + L.x_scales), ws + L.perm,
                               L.offsets - L.perm, stream, loads));
    }
    STATUS_OK(mark(2));
    if (w->fp8) {
        STATUS_OK(fp8_gemm_impl(ws + L.x_perm, reinterpret_cast<float*>(ws + L.x_scales),
                                reinterpret_cast<const uint8_t*>(w->w13), w->w13_scales, offsets, N + 1, R, 2 * I, d,
                                MOE_EPI_SWIGLU_FP8, ws + L.act, reinterpret_cast<float*>(ws + L.act_scales), h_out,
                                stream, gather ? perm_token : nullptr, T * K, T));
        STATUS_OK(mark(3));
        STATUS_OK(fp8_grouped_gemm(ws + L.act, reinterpret_cast<float*>(ws + L.act_scales),
                                   reinterpret_cast<const uint8_t*>(w->w2), w->w2_scales, offsets, N + 1, R, d, I,
                                   MOE_EPI_BF16, ws + L.y, nullptr, stream));
    } else {
        STATUS_OK(bf16_grouped_gemm(reinterpret_cast<uint16_t*>(ws + L.x_perm),
                                    reinterpret_cast<const uint16_t*>(w->w13), offsets, N + 1, R, 2 * I, d,
                                    MOE_EPI_SWIGLU_BF16, ws + L.act, stream));
        STATUS_OK(mark(3));
        STATUS_OK(bf16_grouped_gemm(reinterpret_cast<uint16_t*>(ws + L.act), reinterpret_cast<const uint16_t*>(w->w2),
                                    offsets, N + 1, R, d, I, MOE_EPI_BF16, ws + L.y, stream));
    }
    STATUS_OK(mark(4));
    const uint16_t* y = reinterpret_cast<const uint16_t*>(ws + L.y);
    STATUS_OK(moe_combine(u, y + T * K * int64_t(d), y, gates, dest, T, d, K, R, out, stream));
    STATUS_OK(mark(5));
    if (update_bias) STATUS_OK(moe_bias_update(w->bias, loads, N, T, K, w->gamma, stream));
    STATUS_OK(mark(6));
    return MOE_OK;
}

moe_status moe_layer_forward(const moe_layer_weights* w, const uint16_t* u, int64_t T, uint16_t* out,
                             const moe_layer_outputs* outs, int update_bias, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream) {
    STATUS_OK(check_layer(w));
    REQUIRE(outs && outs->loads, "moe_layer_forward: outputs need a loads buffer");
    REQUIRE(T >= 0 && (T == 0 || (u && out)), "moe_layer_forward: null u/out");
    const LayerWs L = layer_ws(w, T, 0);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_layer_forward: workspace needs %zu bytes, 256-byte aligned", L.total);
    return layer_forward(w, u, T, out, outs, update_bias, reinterpret_cast<uint8_t*>(workspace), L, stream);
}

moe_status moe_layer_forward_host(const moe_layer_weights* w, const uint16_t* u_host, int64_t T, uint16_t* out_host,
                                  const moe_layer_outputs* outs, int update_bias, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream) {
    STATUS_OK(check_layer(w));
    REQUIRE(outs && outs->loads, "moe_layer_forward_host: outputs need a loads buffer");
    REQUIRE(T >= 0 && (T == 0 || (u_host && out_host)), "moe_layer_forward_host: null u/out");
    const LayerWs L = layer_ws(w, T, 1);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_layer_forward_host: workspace needs %zu bytes", L.total);
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    uint16_t* u_dev = reinterpret_cast<uint16_t*>(ws + L.u_dev);
    uint16_t* out_dev = reinterpret_cast<uint16_t*>(ws + L.out_dev);
    const size_t bytes = size_t(T) * w->d * 2;
    CUDA_OK(cudaMemcpyAsync(u_dev, u_host, bytes, cudaMemcpyHostToDevice, stream));
    STATUS_OK(layer_forward(w, u_dev, T, out_dev, outs, update_bias, ws, L, stream));
    CUDA_OK(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, stream));
    return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Pipelined host-buffer layer: consecutive calls overlap their copies with
// each other's compute (two device slots for u and h', two copy streams).
// ---------------------------------------------------------------------------

namespace {

struct HostPipeline {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t h2d_done[2] = {}, compute_done[2] = {}, d2h_done[2] = {};
    bool ready = false;
};
constexpr int kMaxPipeDevices = 64;
std::mutex g_pipe_mutex;
HostPipeline g_pipe[kMaxPipeDevices];

// The current device's copy streams and events, created on first use and kept
// for the life of the process.
moe_status host_pipeline(HostPipeline** out) {
    int dev = 0;
    CUDA_OK(cudaGetDevice(&dev));
    REQUIRE(dev >= 0 && dev < kMaxPipeDevices, "pipelined host call: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipeline& p = g_pipe[dev];
    if (!p.ready) {
        CUDA_OK(cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking));
        CUDA_OK(cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking));
        for (int i = 0; i < 2; ++i) {
            CUDA_OK(cudaEventCreateWithFlags(&p.h2d_done[i], cudaEventDisableTiming));
            CUDA_OK(cudaEventCreateWithFlags(&p.compute_done[i], cudaEventDisableTiming));
            CUDA_OK(cudaEventCreateWithFlags(&p.d2h_done[i], cudaEventDisableTiming));
        }
        p.ready = true;
    }
    *out = &p;
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_layer_host_pipeline_workspace_size(const moe_layer_weights* w, int64_t T) {
    return w ? layer_ws(w, T, 2).total : 0;
}

moe_status moe_layer_forward_host_pipelined(const moe_layer_weights* w, const uint16_t* u_host, int64_t T,
                                            uint16_t* out_host, const moe_layer_outputs* outs, int update_bias,
                                            int slot, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                            void* done_event) {
    STATUS_OK(check_layer(w));
    REQUIRE(outs && outs->loads, "moe_layer_forward_host_pipelined: outputs need a loads buffer");
    REQUIRE(T >= 0 && (T == 0 || (u_host && out_host)), "moe_layer_forward_host_pipelined: null u/out");
    REQUIRE(slot == 0 || slot == 1, "moe_layer_forward_host_pipelined: slot must be 0 or 1");
    REQUIRE(done_event, "moe_layer_forward_host_pipelined: null done event");
    const LayerWs L = layer_ws(w, T, 2);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_layer_forward_host_pipelined: workspace needs %zu bytes", L.total);
    HostPipeline* P = nullptr;
    STATUS_OK(host_pipeline(&P));
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    const size_t bytes = size_t(T) * w->d * 2;
    uint16_t* u_dev = reinterpret_cast<uint16_t*>(ws + L.u_dev + slot * bytes);
    uint16_t* out_dev = reinterpret_cast<uint16_t*>(ws + L.out_dev + slot * bytes);
    cudaEvent_t done = reinterpret_cast<cudaEvent_t>(done_event);
    // 1. copy u in once the compute that last read this slot has finished
    CUDA_OK(cudaStreamWaitEvent(P->h2d, P->compute_done[slot], 0));
    if (bytes) CUDA_OK(cudaMemcpyAsync(u_dev, u_host, bytes, cudaMemcpyHostToDevice, P->h2d));
    CUDA_OK(cudaEventRecord(P->h2d_done[slot], P->h2d));
    // 2. compute on the caller's stream once u is in and this slot's last h' has been copied out
    CUDA_OK(cudaStreamWaitEvent(stream, P->h2d_done[slot], 0));
    CUDA_OK(cudaStreamWaitEvent(stream, P->d2h_done[slot], 0));
    STATUS_OK(layer_forward(w, u_dev, T, out_dev, outs, update_bias, ws, L, stream));
    CUDA_OK(cudaEventRecord(P->compute_done[slot], stream));
    // 3. copy h' out; `done` completes when out_host holds it
    CUDA_OK(cudaStreamWaitEvent(P->d2h, P->compute_done[slot], 0));
    if (bytes) CUDA_OK(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, P->d2h));
    CUDA_OK(cudaEventRecord(P->d2h_done[slot], P->d2h));
    CUDA_OK(cudaEventRecord(done, P->d2h));
    return MOE_OK;
}

}  // extern "C"
