/*
 * moe.h — C ABI of the B300 (sm_103a) DeepSeekMoE layer forward.
 *
 * What the layer computes (DeepSeek-V3 Technical Report, as summarised on
 * learn.ifs.name "DeepSeek-V3 Technical Report" and nlp-lineage.vercel.app
 * "DeepSeek-V3 Technical Report (2024)"):
 *
 *   s_{i,t} = sigmoid(u_t . e_i)          affinity of token t to expert i's centroid
 *   chosen  = top-K of s_{i,t} + b_i       the bias b_i steers the choice only
 *   g_{i,t} = s_{i,t} / sum_chosen s       gates normalised over the chosen experts
 *   h'_t    = u_t + FFN_shared(u_t) + sum_chosen g_{i,t} FFN_i(u_t)
 *   after the step: b_i -= gamma if expert i was overloaded, += gamma if underloaded
 *
 * with every expert FFN a SwiGLU MLP run as FP8 GEMMs: activations scaled per
 * 1x128 tile, weights per 128x128 block, partial sums promoted to FP32 every
 * 128 K-elements where the two scales are applied.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE memory owned by the caller, except in
 *     moe_layer_forward_host, whose u/out are host memory. The library never
 *     allocates or frees device memory; scratch comes from a caller workspace
 *     sized by the matching *_workspace_size function (moe_permute_static
 *     instead uses a fixed array inside the library, see there).
 *   - Calls are asynchronous on `stream` and return synchronously checked
 *     argument errors. Device-side problems (a pipeline wait that ran out of
 *     time, inconsistent group offsets) set a device status word that
 *     moe_get_device_status() reads.
 *   - bf16 is passed as uint16_t bit patterns, OCP FP8 E4M3 as uint8_t,
 *     scales as fp32. Row-major unless stated.
 *   - Activation scales are stored K-block-major: scales[kb * ld + row]
 *     (kb = column / 128). Weight scales are [rows/128][cols/128] row-major.
 *   - Pointers used by vector or TMA loads must be 16-byte aligned; GEMM
 *     outputs (C) 32-byte aligned.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t;   /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size           */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement   */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed                 */
    MOE_ERR_TIMEOUT = 4,       /* device: a bounded pipeline wait gave up    */
    MOE_ERR_WORKSPACE = 5,     /* workspace missing or too small            */
    MOE_ERR_DEVICE_DATA = 6    /* device: offsets/indices out of range       */
} moe_status;

enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1, MOE_DTYPE_E4M3 = 2 };

enum {
    MOE_EPI_BF16 = 0,          /* C = bf16(A B^T)                                         */
    MOE_EPI_SWIGLU_FP8 = 1,    /* C = e4m3 1x128 quant of silu(h_gate) * h_up, + scales   */
    MOE_EPI_SWIGLU_BF16 = 2,   /* C = bf16(silu(h_gate) * h_up)                           */
    MOE_EPI_F32 = 3            /* C = fp32(A B^T)                                         */
};

/* Human-readable text of the last host-side error (thread-local). */
const char* moe_last_error(void);

/* Number of SMs the kernels size their persistent grids for (the current device). */
int moe_num_sms(void);

/*
 * Device status word: synchronises `stream`, returns the worst status any
 * kernel recorded since the last call (MOE_OK if none) and clears it.
 */
moe_status moe_get_device_status(moe_stream_t stream, int* status);

/* ------------------------------------------------------------------------ */
/* FP8 quantisation — learn.ifs.name summary, paragraph on FP8 scaling:      */
/* one scale per 1x128 activation tile and per 128x128 weight block, so an   */
/* outlier only affects its own group. scale = amax/448 (1 for an all-zero    */
/* tile), q = e4m3_rn_satfinite(x / scale), both divisions IEEE fp32.         */
/* ------------------------------------------------------------------------ */

/* x bf16 [rows, cols] (row stride ld_x elements), cols % 128 == 0.
 * q e4m3 [rows, cols] (row stride cols); scales[kb * ld_s + r], ld_s >= rows. */
moe_status fp8_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                           uint8_t* q, float* scales, int64_t ld_s, moe_stream_t stream);

/* w bf16 [rows, cols], cols % 128 == 0 (a last partial row block holds the
 * rows that exist). q e4m3 [rows, cols]; scales [ceil(rows/128)][cols/128]. */
moe_status fp8_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols,
                             uint8_t* q, float* scales, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Routing — learn.ifs.name summary, MoE and bias paragraphs; nlp-lineage    */
/* page, "The notation": chosen iff s + b is among the top K; the bias       */
/* affects only the choice. Ties go to the lower expert index.               */
/* ------------------------------------------------------------------------ */

/* u bf16 [T, d]; centroids [N, d] bf16 or fp32 (centroid_dtype); bias fp32 [N].
 * n_groups = 1: flat top-K. n_groups > 1: experts form n_groups groups of
 * N/n_groups consecutive ids, a group's score is the sum of its two largest
 * s + b, and only the topk_groups best groups (ties: lower group) compete.
 * Outputs: topk_idx int32 [T, K] (ascending expert id per token), gates fp32
 * [T, K] (s / sum s over the chosen), loads int32 [N] (overwritten: tokens
 * per expert), scores fp32 [T, N] (s; may be NULL).
 * Limits: d % 64 == 0, 1 <= K <= 16, K <= N <= 1024, N % 16 == 0 when
 * centroids are fp32 (tensor-core gate), n_groups <= 32. */
size_t moe_route_workspace_size(int64_t T, int d, int N, int centroid_dtype);
moe_status moe_route(const uint16_t* u, int64_t T, int d, const void* centroids, int centroid_dtype,
                     const float* bias, int N, int K, int n_groups, int topk_groups,
                     int32_t* topk_idx, float* gates, int32_t* loads, float* scores,
                     void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_route in two parts, for centroids that stay fixed across calls (the
 * centroids are weights of the layer; only the bias changes between steps).
 * moe_route_prepare_centroids writes the tensor-core operand of the gate once:
 * fp32 centroids split exactly into three bf16 terms (bf16 centroids are
 * copied), zero rows up to a multiple of 256 experts. `prepared` is device
 * memory of moe_route_prepared_centroids_size() bytes, 256-byte aligned,
 * owned by the caller; it must be prepared again if the centroids change.
 * moe_route_prepared then routes from it with the same arguments, outputs and
 * limits as moe_route, and a workspace of moe_route_prepared_workspace_size()
 * bytes (the split-K partial logits only). The two calls give bit-identical
 * results to moe_route. */
size_t moe_route_prepared_centroids_size(int d, int N, int centroid_dtype);
moe_status moe_route_prepare_centroids(const void* centroids, int centroid_dtype, int N, int d,
                                       void* prepared, size_t prepared_bytes, moe_stream_t stream);
size_t moe_route_prepared_workspace_size(int64_t T, int d, int N, int centroid_dtype);
moe_status moe_route_prepared(const uint16_t* u, int64_t T, int d, const void* prepared,
                              int centroid_dtype, const float* bias, int N, int K, int n_groups,
                              int topk_groups, int32_t* topk_idx, float* gates, int32_t* loads,
                              float* scores, void* workspace, size_t workspace_bytes,
                              moe_stream_t stream);

/* Sequence-wise balance statistics of one routing step — learn.ifs.name
 * summary, bias paragraph: beside the bias, only a tiny sequence-wise
 * balancing loss remains, against extreme imbalance inside one sequence. The
 * pages give no formula; the statistic computed here, for each sequence of
 * seq_len consecutive tokens (the last may be shorter, T_s tokens), is
 *   seq_loads[s][i] = pairs (t, k) of the sequence with topk_idx[t][k] == i
 *   seq_prob[s][i]  = (1/T_s) sum_t scores[t][i] / sum_j scores[t][j]
 *   seq_stat[s]     = sum_i (N seq_loads[s][i] / (K T_s)) seq_prob[s][i]
 * (the loss weight is the caller's). scores fp32 [T, N]: the affinities s from
 * moe_route's scores output; topk_idx int32 [T, K] in [0, N). Outputs:
 * seq_loads int32 [S, N], seq_prob fp32 [S, N], seq_stat fp32 [S], S =
 * ceil(T / seq_len). Sums run in a fixed order (reproducible bit for bit).
 * Workspace: moe_route_balance_stats_workspace_size() bytes, 16-byte aligned.
 * An id outside [0, N) is skipped and sets MOE_ERR_DEVICE_DATA. */
size_t moe_route_balance_stats_workspace_size(int64_t T, int N, int64_t seq_len);
moe_status moe_route_balance_stats(const float* scores, const int32_t* topk_idx, int64_t T, int N, int K,
                                   int64_t seq_len, int32_t* seq_loads, float* seq_prob, float* seq_stat,
                                   void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Permutation — the single-GPU form of the dispatch step (learn.ifs.name    */
/* summary, paragraph on all-to-all dispatch/combine): a stable counting     */
/* sort of the (token, expert) pairs by expert, tokens ascending within one  */
/* expert, no pair dropped (nlp-lineage page, load-balancing item).          */
/* ------------------------------------------------------------------------ */

/* x bf16 [T, d]; topk_idx int32 [T, K] with entries in [0, N).
 * out_dtype MOE_DTYPE_BF16: x_perm bf16 rows; MOE_DTYPE_E4M3: x_perm e4m3
 * rows quantised per 1x128 tile, scales[kb * R + row] with R the row count.
 * with_shared != 0 appends rows T*K .. T*K+T-1 = x[0..T-1] (the shared
 * expert's group), so R = T*K + T and offsets has N + 2 entries; else
 * R = T*K and offsets has N + 1 entries (offsets[i] = first row of expert i).
 * perm_token int32 [T*K]: source token of each routed row;
 * dest_row int32 [T, K]: row of each (token, k). d % 128 == 0. */
size_t moe_permute_workspace_size(int64_t T, int N);
moe_status moe_permute(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K,
                       int out_dtype, int with_shared, int32_t* offsets, int32_t* perm_token,
                       int32_t* dest_row, void* x_perm, float* x_perm_scales,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_permute without a workspace. The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory, such as code
 * whose device memory all belongs to another allocator it cannot ask for a
 * buffer, or code that must not allocate once running (cudaMalloc can
 * synchronise the device or fail under memory pressure).
 *
 * Same arguments, outputs and rules as moe_permute. The scratch (per-chunk
 * expert histograms) is a 4 MiB array inside the library, held on every GPU
 * that loads the library until the process exits. Limit: ceil(T/32)*N + N
 * <= 1,048,576 (e.g. N = 256 allows T <= 131,040); larger sizes return
 * MOE_ERR_WORKSPACE without launching anything. Calls no allocator.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and caches it. Make that first call
 * before any stream capture. The cached address belongs to the CUDA context
 * of that first call: it is dropped when a launch fails, but it does not
 * survive cudaDeviceReset, after which this entry point must not be called
 * again in the same process.
 *
 * Every call on a device shares the one array. The kernels write each
 * scratch entry before reading it, so nothing must start at zero and the
 * previous call's contents do not matter. Calls that overlap on the GPU
 * (different streams, no ordering between them) race on the array and give
 * wrong results: order them on one stream, or use moe_permute. */
moe_status moe_permute_static(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K,
                              int out_dtype, int with_shared, int32_t* offsets, int32_t* perm_token,
                              int32_t* dest_row, void* x_perm, float* x_perm_scales, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped GEMMs — learn.ifs.name summary, paragraphs on FP8 tiles and on     */
/* promotion: every 128 K-elements the partial sums go to FP32 and the       */
/* per-group scales are applied there.                                       */
/* ------------------------------------------------------------------------ */

/* For each group g (rows group_offsets[g] .. group_offsets[g+1]-1 of A):
 *   C[rows] = epilogue( sum_kb sa[kb][row] * sb[g][n/128][kb] * (A[row, kb] . B[g][n, kb]) )
 * A e4m3 [M_total, Kd]; sa fp32 [Kd/128][M_total]; B e4m3 [G][Nd][Kd] (K
 * contiguous); sb fp32 [G][Nd/128][Kd/128]; group_offsets int32 [G+1] in
 * DEVICE memory, non-decreasing from 0 to <= M_total.
 * MOE_EPI_BF16: C bf16 [M_total, Nd].
 * MOE_EPI_SWIGLU_FP8: B's rows alternate per 128 between the gate and the up
 * projection (rows 256j..256j+127 = W1 rows 128j.., rows 256j+128.. = W3 rows
 * 128j..); C e4m3 [M_total, Nd/2] = 1x128 quant of silu(h1) * h3 with scales
 * c_scales[j * M_total + row] (j = output column / 128).
 * Limits: Kd % 128 == 0, Nd % 256 == 0, G <= 1024. Rows past a group's end are
 * never written. */
moe_status fp8_grouped_gemm(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                            const int32_t* group_offsets, int G, int64_t M_total, int Nd, int Kd,
                            int epilogue, void* C, float* c_scales, moe_stream_t stream);

/* Same grouping with bf16 A [M_total, Kd], B [G][Nd][Kd] and FP32
 * accumulation over the whole K (no scales). epilogue MOE_EPI_BF16 (C bf16
 * [M_total, Nd]), MOE_EPI_SWIGLU_BF16 (C bf16 [M_total, Nd/2], rows of B
 * interleaved as above) or MOE_EPI_F32 (C fp32 [M_total, Nd]).
 * Limits: Kd % 64 == 0, Nd % 256 == 0, G <= 1024. */
moe_status bf16_grouped_gemm(const uint16_t* A, const uint16_t* B, const int32_t* group_offsets,
                             int G, int64_t M_total, int Nd, int Kd, int epilogue, void* C,
                             moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Combine — nlp-lineage page, "The notation":                               */
/*   h'_t = u_t + y_shared_t + sum_k g_{t,k} y_{dest_row[t,k]}               */
/* accumulated in fp32 in that order (k ascending), stored as bf16.          */
/* ------------------------------------------------------------------------ */

/* u bf16 [T, d]; y_shared bf16 [T, d] or NULL; y_perm bf16 [R, d];
 * gates fp32 [T, K]; dest_row int32 [T, K] in [0, R); out bf16 [T, d].
 * d % 8 == 0. */
moe_status moe_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y_perm,
                       const float* gates, const int32_t* dest_row, int64_t T, int d, int K,
                       int64_t R, uint16_t* out, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Bias update — learn.ifs.name summary, bias paragraph; nlp-lineage page,   */
/* load-balancing item. Overloaded = load above the mean T*K/N (compared as  */
/* load*N vs T*K): b -= gamma; below: b += gamma; equal: unchanged.          */
/* ------------------------------------------------------------------------ */

moe_status moe_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma,
                           moe_stream_t stream);

/* Self-test of the device-side failure detection; the paper has no
 * counterpart. Launches one thread that waits, with the pipelines' bounded
 * wait and a limit of limit_ns (at most 1 s), on an mbarrier that nothing
 * arrives on. It gives up, records MOE_ERR_TIMEOUT in the device status word
 * (read it with moe_get_device_status) and returns; the CUDA context stays
 * usable. */
moe_status moe_selftest_wait_timeout(int64_t limit_ns, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The whole layer, composed from the calls above.                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    int d, N, K, I;            /* hidden, routed experts, experts per token, SwiGLU width   */
    int n_groups, topk_groups; /* routing groups (1, 1 = flat)                              */
    float gamma;               /* bias step                                                 */
    int fp8;                   /* 1: e4m3 weights + scales; 0: bf16 weights, no scales      */
    const void* centroids;     /* [N, d] */
    int centroid_dtype;        /* MOE_DTYPE_F32 or MOE_DTYPE_BF16                           */
    float* bias;               /* [N] fp32, updated in place when update_bias != 0          */
    const void* w13;           /* [N+1][2I][d], gate/up rows interleaved per 128; expert N = shared */
    const float* w13_scales;   /* [N+1][2I/128][d/128] (fp8 only)                           */
    const void* w2;            /* [N+1][d][I]                                               */
    const float* w2_scales;    /* [N+1][d/128][I/128] (fp8 only)                            */
    const void* centroids_prepared; /* NULL, or the output of moe_route_prepare_centroids for
                                       `centroids` (then the layer routes from it)           */
    int dispatch;              /* FP8 layers: MOE_DISPATCH_SCATTER (0) or MOE_DISPATCH_GATHER   */
} moe_layer_weights;

/* How an FP8 layer hands the tokens to grouped GEMM 1 (the dispatch):
 *   MOE_DISPATCH_SCATTER  moe_permute writes every (token, k) row, quantised, to
 *                         its place in the expert-grouped rows; GEMM 1 reads
 *                         those rows by TMA.
 *   MOE_DISPATCH_GATHER   the tokens are quantised once (fp8_quant_1x128), the
 *                         permutation moves no rows, and GEMM 1 gathers each
 *                         row of its A operand from the quantised tokens by
 *                         perm_token (cp.async): the grouped rows are never
 *                         written. The results are the same bits.
 * bf16 layers always scatter. */
enum { MOE_DISPATCH_SCATTER = 0, MOE_DISPATCH_GATHER = 1 };

/* Optional outputs of one forward (any may be NULL except loads). */
typedef struct {
    int32_t* topk_idx;         /* [T, K] */
    float* gates;              /* [T, K] */
    int32_t* loads;            /* [N], required */
    /* NULL, or MOE_LAYER_STAGES + 1 cudaEvent_t recorded on `stream` before the
     * first stage and after each stage (route, permute, GEMM 1, GEMM 2,
     * combine, bias update) — for timing the stages inside a run. */
    void* const* stage_events;
} moe_layer_outputs;

#define MOE_LAYER_STAGES 6

size_t moe_layer_workspace_size(const moe_layer_weights* w, int64_t T);

/* h' for T tokens: u bf16 [T, d] -> out bf16 [T, d] (device), then the bias
 * update from this step's loads when update_bias != 0. Launch sequence:
 * route, permute (with FP8 quantisation of the rows when fp8; it also counts
 * the loads), grouped GEMM 1 with SwiGLU, grouped GEMM 2, combine, bias
 * update. */
moe_status moe_layer_forward(const moe_layer_weights* w, const uint16_t* u, int64_t T, uint16_t* out,
                             const moe_layer_outputs* outs, int update_bias,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* As moe_layer_forward with u_host / out_host in HOST memory (pinned for
 * speed): copies u in, runs the layer, copies h' back, all on `stream`.
 * The device copies of u and out live in the workspace
 * (moe_layer_host_workspace_size). */
size_t moe_layer_host_workspace_size(const moe_layer_weights* w, int64_t T);
moe_status moe_layer_forward_host(const moe_layer_weights* w, const uint16_t* u_host, int64_t T,
                                  uint16_t* out_host, const moe_layer_outputs* outs, int update_bias,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Pipelined form of moe_layer_forward_host for a stream of batches: the
 * host-to-device copy of one call and the device-to-host copy of the previous
 * call run on two copy streams of the library while a call computes on
 * `stream`, so copies and compute of consecutive calls overlap.
 * Alternate `slot` (0, 1, 0, 1, ...) between consecutive calls that share one
 * workspace (sized by moe_layer_host_pipeline_workspace_size, same w and T).
 * `done_event` (a cudaEvent_t the caller created) is recorded once h' is in
 * out_host; a synchronisation of `stream` alone does NOT cover that copy.
 * out_host may be read, and u_host overwritten, once `done_event` has
 * completed. The copy streams and events are created on the first call on a
 * device and live until the process exits. They are shared by every
 * pipelined call on that device: calls from different workspaces stay
 * correct but wait on one another's copies of the same slot index. */
size_t moe_layer_host_pipeline_workspace_size(const moe_layer_weights* w, int64_t T);
moe_status moe_layer_forward_host_pipelined(const moe_layer_weights* w, const uint16_t* u_host, int64_t T,
                                            uint16_t* out_host, const moe_layer_outputs* outs, int update_bias,
                                            int slot, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                            void* done_event);

/* ------------------------------------------------------------------------ */
/* Training: the layer's backward pass and one SGD step.                      */
/* ------------------------------------------------------------------------ */
/* Sources: nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)",
 * "The idea", FP8-training item (the heavy products of training run in
 * 8-bit floating point, scaled in small tiles and blocks) and "The notation"
 * (the layer formula); learn.ifs.name "DeepSeek-V3 Technical Report", DualPipe
 * paragraph (each layer has a forward and a backward chunk: dispatch, MLP,
 * combine) and bias paragraph (the bias moves after each training step).
 * Readings (the pages give no formula for the backward): the gradient of
 *   h'_t = u_t + FFN_shared(u_t) + sum_k g_{t,k} FFN_{idx(t,k)}(u_t)
 * with the expert choice held fixed and every quantisation or bf16 rounding
 * passed straight through:
 *   combine   dY_row(t,k) = g_{t,k} G_t (fp32), dY_shared,t = G_t,
 *             dg_{t,k} = G_t . y_row(t,k)        (G = dL/dh', bf16)
 *   expert    dA = dY W2 and dX = dH W13 on the tensor cores, FP8 operands:
 *             dY and dH per 1x128 tile (the tile rule is scale-invariant, so a
 *             routed row's dY = g G_t takes G_t's codes and g times its
 *             scales: no fp32 rounding of g G_t), the weights' forward 128x128 blocks
 *             transposed; dA, dH and dX stored in bf16; dH from the stored
 *             bf16 products H of the forward (dh1 = dA h3 s (1 + h1 (1 - s)),
 *             dh3 = dA h1 s, s = sigmoid(h1));
 *             dW2 = dY^T A and dW13 = dH^T X contract over the expert's own
 *             tokens: both operands quantised per (128 tokens, column), A
 *             recomputed in fp32 from H, X = u of the rows; fp32 out;
 *   gates     S = sum_k s_k, c = sum_k g_k dg_k, dz_k = (dg_k - c) / S s'(z_k), with the
 *             sigmoid's derivative s (1 - s) evaluated from the logit as
 *             e^-|z| / (1 + e^-|z|)^2 (no cancellation in 1 - s when s is near 1);
 *   tokens    du_t = G_t + dX_shared,t + sum_k dX_row(t,k) + sum_k dz_k e_idx(t,k)  (bf16);
 *   centroids de_i = sum over the (t, k) routed to i of dz_{t,k} u_t  (fp32);
 *   bias      no gradient: it moves by the load rule after the step.
 * The training step is plain SGD on fp32 master weights, w <- fl32(w -
 * fl32(lr dw)), after which the FP8 weights are quantised again. FP8 layers
 * only; I must be a multiple of 256. */

/* W13 and W2 of a FP8 layer quantised per 128x128 block, transposed (codes and
 * scale grid), for the backward's products dA = dY W2 and dX = dH W13. */
typedef struct {
    uint8_t* w13t;             /* [N+1][d][2I] e4m3 */
    float* w13t_scales;        /* [N+1][d/128][2I/128] */
    uint8_t* w2t;              /* [N+1][I][d] */
    float* w2t_scales;         /* [N+1][I/128][d/128] */
} moe_layer_weights_t;

/* Gradients written by moe_layer_backward (all device memory). */
typedef struct {
    float* dw13;               /* [N+1][2I][d] fp32, rows in W13's interleaved order; required */
    float* dw2;                /* [N+1][d][I] fp32; required */
    float* dcentroids;         /* [N][d] fp32; required */
    float* dz;                 /* [T, K] fp32 gradient of the chosen experts' logits; optional */
    /* NULL, or MOE_BACKWARD_STAGES + 1 cudaEvent_t recorded on `stream` before
     * the first stage and after each stage of moe_layer_backward (combine
     * backward, GEMM dA, SwiGLU backward, GEMM dX, gates + du + centroid
     * gradient, weight-gradient operands, GEMM dW2, GEMM dW13). */
    void* const* stage_events;
} moe_layer_grads;

#define MOE_BACKWARD_STAGES 8

/* fp32 master copies of the FP8 layer's expert weights (training step). */
typedef struct {
    float* w13;                /* [N+1][2I][d], W13's interleaved row order */
    float* w2;                 /* [N+1][d][I] */
} moe_layer_masters;

/* The workspace of a training step: the forward's, plus what the backward
 * keeps (H, the affinities) and its own intermediates. One workspace serves
 * moe_layer_forward_train and the moe_layer_backward that follows it. */
size_t moe_layer_train_workspace_size(const moe_layer_weights* w, int64_t T);

/* moe_layer_forward that also keeps, in the workspace, what the backward
 * reads: the affinities s and gate logits z [T, N] and GEMM 1's products
 * H [T*K+T, 2I] in bf16. */
moe_status moe_layer_forward_train(const moe_layer_weights* w, const uint16_t* u, int64_t T, uint16_t* out,
                                   const moe_layer_outputs* outs, int update_bias, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream);

/* Backward of the moe_layer_forward_train call that last used `workspace`
 * (same w, u and T): dout = dL/dh' bf16 [T, d] -> du bf16 [T, d] and grads.
 * Launch sequence: combine backward, FP8 grouped GEMM dA, SwiGLU backward,
 * FP8 grouped GEMM dX, gate backward and du, centroid gradient, the
 * weight-gradient operands, two FP8 weight-gradient GEMMs. */
moe_status moe_layer_backward(const moe_layer_weights* w, const moe_layer_weights_t* wt, const uint16_t* u,
                              int64_t T, const uint16_t* dout, uint16_t* du, const moe_layer_grads* grads,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* One training step: moe_layer_forward_train with the bias update, the
 * backward, then SGD with learning rate lr on m's masters and on the fp32
 * centroids (w->centroid_dtype must be MOE_DTYPE_F32), re-quantisation of
 * w13/w2 (+ scales) and of wt from the new masters, and, when
 * w->centroids_prepared is set, the prepared centroids again. Updates in
 * place: w->w13, w->w13_scales, w->w2, w->w2_scales, w->centroids,
 * w->centroids_prepared, w->bias, wt's arrays and m's masters. */
moe_status moe_layer_train_step(const moe_layer_weights* w, const moe_layer_weights_t* wt,
                                const moe_layer_masters* m, const uint16_t* u, int64_t T, const uint16_t* dout,
                                float lr, uint16_t* out, uint16_t* du, const moe_layer_outputs* outs,
                                const moe_layer_grads* grads, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/* Named buffers of the training workspace (for tests and inspection):
 * byte offset and size of `which` for this w and T, or MOE_ERR_INVALID_ARG. */
enum {
    MOE_TRAIN_H = 0,           /* bf16 [R, 2I], R = T*K + T: GEMM 1's products */
    MOE_TRAIN_SCORES = 1,      /* fp32 [T, N] affinities */
    MOE_TRAIN_DG = 2,          /* fp32 [T, K] */
    MOE_TRAIN_DA = 3,          /* bf16 [R, I] */
    MOE_TRAIN_DH = 4,          /* bf16 [R, 2I] */
    MOE_TRAIN_DX = 5,          /* bf16 [R, d] */
    MOE_TRAIN_OFFSETS = 6,     /* int32 [N+2] row offsets of the groups */
    MOE_TRAIN_PERM_TOKEN = 7,  /* int32 [T*K] */
    MOE_TRAIN_DEST_ROW = 8,    /* int32 [T, K] */
    MOE_TRAIN_Y = 9,           /* bf16 [R, d] expert outputs */
    MOE_TRAIN_KOFS = 10,       /* int32 [N+2] 128-row block offsets of the weight-gradient K layout */
    MOE_TRAIN_DY_Q = 11,       /* e4m3 [R, d] the operand dY of dA = dY W2 */
    MOE_TRAIN_DY_S = 12,       /* fp32 [d/128, R] its 1x128 scales */
    MOE_TRAIN_DH_Q = 13,       /* e4m3 [R, 2I] the operand dH of dX = dH W13 */
    MOE_TRAIN_DH_S = 14,       /* fp32 [2I/128, R] its 1x128 scales */
    MOE_TRAIN_ROW_GATE = 15,   /* fp32 [R] the gate of each row (1 for the shared expert's) */
    MOE_TRAIN_LOGITS = 16      /* fp32 [T, N] the gate logits z (s = sigmoid(z)) */
};
moe_status moe_layer_train_buffer(const moe_layer_weights* w, int64_t T, int which, size_t* offset,
                                  size_t* bytes);

/* FP8 weight-gradient GEMM, grouped along K: for each group g,
 *   C[g][m][n] = sum over its 128-K blocks kb of
 *                sa[kb][m] * sb[kb][n] * sum_{k in kb} A[m][k] * B[n][k]
 * (each block's partial sum promoted in fp32 with its scales, as in the
 * forward's products). A e4m3 [M][Kp], B e4m3 [Nd][Kp] (K contiguous),
 * sa fp32 [Kp/128][M], sb fp32 [Kp/128][Nd], kofs int32 [G+1] device: group
 * g owns K blocks kofs[g] .. kofs[g+1]-1 (non-decreasing, kofs[0] = 0,
 * kofs[G] <= Kp/128; a group with no blocks gets zeros). C fp32 [G][M][Nd].
 * M % 128 == 0, Nd % 256 == 0, Kp % 128 == 0. Bad offsets set
 * MOE_ERR_DEVICE_DATA in the device status and write nothing. */
moe_status fp8_grouped_gemm_wgrad(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                                  const int32_t* kofs, int G, int M, int Nd, int64_t Kp, float* C,
                                  moe_stream_t stream);

/* 128x128-block E4M3 codes and their scales transposed, per group:
 * q [G][rows][cols], s [G][rows/128][cols/128] -> qt [G][cols][rows],
 * st [G][cols/128][rows/128]. rows, cols multiples of 128. */
moe_status fp8_transpose_128x128(const uint8_t* q, const float* s, int G, int rows, int cols, uint8_t* qt,
                                 float* st, moe_stream_t stream);

/* SGD on an fp32 master [G][rows][cols] and its 128x128 re-quantisation:
 * w <- fl32(w - fl32(lr * grad)) (two roundings), then per block
 * scale = amax/448 and q = e4m3(w / scale), stored as is (q [G][rows][cols],
 * s [G][rows/128][cols/128]) and transposed (qt [G][cols][rows],
 * st [G][cols/128][rows/128]). rows, cols multiples of 128. */
moe_status moe_sgd_requant_128x128(float* w, const float* grad, int G, int rows, int cols, float lr, uint8_t* q,
                                   float* s, uint8_t* qt, float* st, moe_stream_t stream);

/* w <- fl32(w - fl32(lr * grad)) for n fp32 values. */
moe_status moe_sgd_f32(float* w, const float* grad, int64_t n, float lr, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
