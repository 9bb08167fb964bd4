/*
 * FP64 CPU oracle for the DeepSeekMoE layer: forward, backward, training step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this file's library. It is a
 * plain, slow, obviously correct restatement of what the layer computes, and
 * shares no code, header, table or constant with the CUDA library.
 *
 * Sources (the DeepSeek-V3 Technical Report as summarised on the web):
 *   [moe]     learn.ifs.name "DeepSeek-V3 Technical Report", paragraph on the
 *             shared expert and the 256 routed experts: top-8 by sigmoid
 *             affinity to each expert's centroid, gates normalised over the
 *             chosen experts, each token sent to at most 4 nodes.
 *   [bias]    same page, paragraph on the per-expert bias: added to the
 *             affinity for top-K routing only; after each step lowered by
 *             gamma for an overloaded expert and raised for an underloaded one.
 *   [tiles]   same page, paragraph on FP8 scaling: activations per 1x128 tile
 *             (per token, per 128 channels), weights per 128x128 block.
 *   [promote] same page, paragraph on accumulation: every 128 elements the
 *             partial sums are promoted to FP32 and the per-group scales are
 *             applied there.
 *   [formula] nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)",
 *             section "The idea", "The notation":
 *             h'_t = u_t + sum_shared FFN_i(u_t) + sum_routed g_it FFN_i(u_t);
 *             an expert is chosen if s_it + b_i is among the top 8; the bias
 *             affects only the choice, not g.
 *   [nodrop]  same page, "The idea", load-balancing item: no token is dropped.
 *   [seqloss] learn.ifs.name, bias paragraph: beside the bias, only a tiny
 *             sequence-wise balancing loss remains, against extreme
 *             imbalance inside one sequence.
 *   [train]   nlp-lineage.vercel.app, "The idea", FP8-training item: most
 *             heavy calculations of training run in 8-bit floating point,
 *             scaled in small tiles and blocks; learn.ifs.name, DualPipe
 *             paragraph: each layer has forward and backward chunks; bias
 *             paragraph: the bias moves after each training step.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   affinity s = 1/(1+exp(-u.e_i)); gates g = s/sum(s chosen) with factor 1;
 *   ties go to the lower expert (group) index; FP8 is OCP E4M3 with round to
 *   nearest even, saturating at 448; tile scale = amax/448 as an fp32
 *   division (1 for an all-zero tile) and q = e4m3(x / scale) as an fp32
 *   division; expert FFN = W2 (silu(W1 x) * W3 x); "overloaded" means a load
 *   above the mean T*K/N, "underloaded" below it. The sequence-wise
 *   balance statistic of a sequence of T_s tokens is sum_i f_i * P_i with
 *   f_i = N * (pairs routed to i) / (K * T_s) and P_i the mean over the
 *   sequence of s_i / sum_j s_j (affinities normalised over all N experts);
 *   the loss weight is the caller's.
 *
 * Every floating-point sum below runs in FP64, in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
double oracle_bf16_value(uint16_t b)
{
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

/* Round x to bf16 (8 significant bits) with ties to even, directly from
 * double (no intermediate fp32 rounding). Finite inputs below 2^127 only. */
uint16_t oracle_bf16_round(double x)
{
    if (x == 0.0) {
        return signbit(x) ? 0x8000u : 0u;
    }
    int e;
    double m = frexp(fabs(x), &e);            /* |x| = m * 2^e, m in [0.5, 1) */
    int shift = 8;                            /* keep 8 significant bits      */
    if (e - 1 < -126) shift = 8 - (-126 - (e - 1));   /* bf16 subnormals    */
    double scaled = ldexp(m, shift);
    double fl = floor(scaled);
    double frac = scaled - fl;
    double r;
    if (frac > 0.5) r = fl + 1.0;
    else if (frac < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double y = ldexp(r, e - shift);
    float f = (float)y;                       /* exact: y has <= 8 bits     */
    uint32_t w;
    memcpy(&w, &f, 4);
    uint16_t h = (uint16_t)(w >> 16);
    return signbit(x) ? (uint16_t)(h | 0x8000u) : h;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinity.
 * Largest finite magnitude 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

static double g_e4m3_pos[127];   /* values of codes 0..126, ascending */
static double g_e4m3_all[256];
static int g_tables_ready = 0;

static void tables_init(void)
{
    if (g_tables_ready) return;
    for (int c = 0; c < 127; ++c) g_e4m3_pos[c] = oracle_e4m3_value((uint8_t)c);
    for (int c = 0; c < 256; ++c) g_e4m3_all[c] = oracle_e4m3_value((uint8_t)c);
    g_tables_ready = 1;
}

void oracle_init(void) { tables_init(); }

/* Nearest E4M3 value to v, ties to the even code (mantissa LSB 0),
 * magnitudes beyond 448 saturate to 448, the sign of v is kept (also for
 * zero). Found by binary search over the 127 non-negative finite codes. */
uint8_t oracle_e4m3_encode(float v)
{
    tables_init();
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 126);
    int lo = 0, hi = 126;                 /* invariant: pos[lo] <= a < pos[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_e4m3_pos[mid] <= a) lo = mid; else hi = mid;
    }
    double dlo = a - g_e4m3_pos[lo], dhi = g_e4m3_pos[hi] - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | c);
}

/* Distance from v to the nearest point where the E4M3 rounding of v would
 * change (a midpoint between two adjacent codes of the same sign, or zero),
 * in the units of v. Used to tell which codes another correct fp32
 * computation could round the other way. */
double oracle_e4m3_boundary_distance(float v)
{
    tables_init();
    double a = fabs((double)v);
    if (a >= 448.0) return a - 0.5 * (g_e4m3_pos[125] + g_e4m3_pos[126]);
    double best = a;  /* distance to zero, where the sign bit would change */
    for (int c = 0; c < 126; ++c) {
        double mid = 0.5 * (g_e4m3_pos[c] + g_e4m3_pos[c + 1]);
        double dd = fabs(a - mid);
        if (dd < best) best = dd;
    }
    return best;
}

/* Element-wise forms of the two conversions above, for arrays. */
void oracle_bf16_round_array(const double* x, int64_t n, uint16_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    tables_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------ */
/* FP8 quantisation [tiles]                                                 */
/* ------------------------------------------------------------------------ */

/* One tile: scale = amax/448 (fp32 division; 1 when amax is 0), then
 * q = e4m3(x / scale) with the division in fp32. `vals` are fp32 values. */
static float quant_tile(const float* vals, int64_t n, int64_t stride, uint8_t* q, int64_t qstride)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(vals[i * stride]);
        if (a > amax) amax = a;
    }
    float sc = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = vals[i * stride] / sc;
        q[i * qstride] = oracle_e4m3_encode(v);
    }
    return sc;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, 4);
    return f;
}

/* Activations: one scale per (row, 128 consecutive columns).
 * x bf16 [rows, cols] row-major, cols % 128 == 0.
 * q [rows, cols], scales [rows, cols/128] row-major. */
void oracle_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, float* scales)
{
    tables_init();
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float buf[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) buf[i] = bf16_to_float(x[r * cols + b * 128 + i]);
            scales[r * nb + b] = quant_tile(buf, 128, 1, q + r * cols + b * 128, 1);
        }
    }
}

/* Same tile rule on fp32 input (the intermediate activation of the FFN). */
void oracle_quant_1x128_f32(const float* x, int64_t rows, int64_t cols, uint8_t* q, float* scales)
{
    tables_init();
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            scales[r * nb + b] = quant_tile(x + r * cols + b * 128, 128, 1, q + r * cols + b * 128, 1);
}

/* Weights: one scale per 128x128 block. w bf16 [rows, cols] row-major,
 * cols % 128 == 0; a last partial block of rows holds the rows that exist.
 * q [rows, cols], scales [ceil(rows/128), cols/128] row-major. */
void oracle_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, float* scales)
{
    tables_init();
    int64_t nbr = (rows + 127) / 128, nbc = cols / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t br = 0; br < nbr; ++br) {
        int64_t r0 = br * 128, r1 = r0 + 128 < rows ? r0 + 128 : rows;
        float* buf = (float*)malloc(sizeof(float) * 128 * 128);
        uint8_t* qb = (uint8_t*)malloc(128 * 128);
        for (int64_t bc = 0; bc < nbc; ++bc) {
            int64_t n = 0;
            for (int64_t r = r0; r < r1; ++r)
                for (int i = 0; i < 128; ++i) buf[n++] = bf16_to_float(w[r * cols + bc * 128 + i]);
            float sc = quant_tile(buf, n, 1, qb, 1);
            scales[br * nbc + bc] = sc;
            n = 0;
            for (int64_t r = r0; r < r1; ++r)
                for (int i = 0; i < 128; ++i) q[r * cols + bc * 128 + i] = qb[n++];
        }
        free(buf);
        free(qb);
    }
}

/* ------------------------------------------------------------------------ */
/* Routing [moe] [bias] [formula] [nodrop]                                  */
/* ------------------------------------------------------------------------ */

typedef struct { double key; int id; } ranked_t;

/* Descending key, then ascending id: a total order, so ties go to the lower id. */
static int cmp_ranked(const void* pa, const void* pb)
{
    const ranked_t* a = (const ranked_t*)pa;
    const ranked_t* b = (const ranked_t*)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

static int cmp_int(const void* pa, const void* pb)
{
    int a = *(const int*)pa, b = *(const int*)pb;
    return (a > b) - (a < b);
}

/*
 * For every token t:
 *   z_i = sum_j u[t,j] * e[i,j]        (centroids fp32 or bf16; FP64 sum)
 *   s_i = 1 / (1 + exp(-z_i))          (sigmoid affinity)
 *   key_i = s_i + b_i                  (bias for the choice only)
 *   if n_groups > 1: the N experts form n_groups groups of N/n_groups
 *     consecutive ids; a group's score is the sum of its two largest keys;
 *     only experts of the topk_groups best groups may be chosen
 *   chosen = the K allowed experts with the largest keys (ties: lower id),
 *            reported in ascending id order
 *   g_k = s_{chosen k} / sum_k s_{chosen k}   (raw affinities, no bias)
 * near_tie[t] = 1 when the K-th and (K+1)-th allowed keys, or the last kept
 * and first dropped group scores, are closer than delta: there a correct
 * fp32 computation may pick a different set.
 * loads[i] = number of tokens that chose expert i (every token gets K).
 */
void oracle_route(const uint16_t* u, int64_t T, int64_t d,
                  const float* cent_f32, const uint16_t* cent_bf16,
                  const float* bias, int N, int K, int n_groups, int topk_groups,
                  double delta, int32_t* topk_idx, double* gates, double* s_out,
                  double* key_gap, int32_t* loads, int32_t* near_tie)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < T; ++t) {
        double* s = (double*)malloc(sizeof(double) * N);
        double* key = (double*)malloc(sizeof(double) * N);
        ranked_t* r = (ranked_t*)malloc(sizeof(ranked_t) * N);
        int* allowed = (int*)malloc(sizeof(int) * N);
        int chosen[64];
        for (int i = 0; i < N; ++i) {
            double z = 0.0;
            for (int64_t j = 0; j < d; ++j) {
                double uj = oracle_bf16_value(u[t * d + j]);
                double eij = cent_f32 ? (double)cent_f32[(int64_t)i * d + j]
                                      : oracle_bf16_value(cent_bf16[(int64_t)i * d + j]);
                z += uj * eij;
            }
            s[i] = 1.0 / (1.0 + exp(-z));
            key[i] = s[i] + (double)bias[i];
            if (s_out) s_out[t * N + i] = s[i];
        }
        double gap = INFINITY;
        for (int i = 0; i < N; ++i) allowed[i] = 1;
        if (n_groups > 1) {
            int per = N / n_groups;
            ranked_t gr[1024];
            for (int g = 0; g < n_groups; ++g) {
                for (int k = 0; k < per; ++k) { r[k].key = key[g * per + k]; r[k].id = g * per + k; }
                qsort(r, per, sizeof(ranked_t), cmp_ranked);
                gr[g].key = r[0].key + r[1].key;
                gr[g].id = g;
            }
            qsort(gr, n_groups, sizeof(ranked_t), cmp_ranked);
            for (int i = 0; i < N; ++i) allowed[i] = 0;
            for (int q = 0; q < topk_groups; ++q)
                for (int k = 0; k < per; ++k) allowed[gr[q].id * per + k] = 1;
            if (topk_groups < n_groups) gap = gr[topk_groups - 1].key - gr[topk_groups].key;
        }
        int n = 0;
        for (int i = 0; i < N; ++i)
            if (allowed[i]) { r[n].key = key[i]; r[n].id = i; ++n; }
        qsort(r, n, sizeof(ranked_t), cmp_ranked);
        if (n > K) {
            double g2 = r[K - 1].key - r[K].key;
            if (g2 < gap) gap = g2;
        }
        for (int k = 0; k < K; ++k) chosen[k] = r[k].id;
        qsort(chosen, K, sizeof(int), cmp_int);
        double den = 0.0;
        for (int k = 0; k < K; ++k) den += s[chosen[k]];
        for (int k = 0; k < K; ++k) {
            topk_idx[t * K + k] = chosen[k];
            gates[t * K + k] = s[chosen[k]] / den;
        }
        if (key_gap) key_gap[t] = gap;
        near_tie[t] = gap < delta;
        free(s); free(key); free(r); free(allowed);
    }
    for (int i = 0; i < N; ++i) loads[i] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) loads[topk_idx[t * K + k]] += 1;
}

/* ------------------------------------------------------------------------ */
/* Permutation into per-expert buffers (the single-GPU form of the          */
/* all-to-all dispatch): a stable counting sort by expert id.               */
/* ------------------------------------------------------------------------ */

/* offsets[i] = sum of loads of experts < i (offsets[N] = T*K); rows of
 * expert i follow in ascending token order: perm_token[row] = t and
 * dest_row[t,k] = row of the pair (t, topk_idx[t,k]). */
void oracle_permute(const int32_t* topk_idx, int64_t T, int N, int K,
                    int32_t* offsets, int32_t* perm_token, int32_t* dest_row)
{
    int64_t* count = (int64_t*)calloc((size_t)N, sizeof(int64_t));
    int64_t* fill = (int64_t*)calloc((size_t)N, sizeof(int64_t));
    for (int64_t p = 0; p < T * K; ++p) count[topk_idx[p]] += 1;
    offsets[0] = 0;
    for (int i = 0; i < N; ++i) offsets[i + 1] = (int32_t)(offsets[i] + count[i]);
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[t * K + k];
            int64_t row = offsets[e] + fill[e]++;
            perm_token[row] = (int32_t)t;
            dest_row[t * K + k] = (int32_t)row;
        }
    free(count);
    free(fill);
}

/* ------------------------------------------------------------------------ */
/* Expert GEMMs [tiles] [promote]                                           */
/* ------------------------------------------------------------------------ */

/*
 * C[m,n] = sum over 128-wide K blocks kb of
 *            sa[m,kb] * sb[n/128,kb] * sum_{k in kb} qa[m,k] * qb[n,k]
 * with qa, qb the E4M3 values: every block's partial sum is scaled and added
 * in full precision. In FP64 each product and each block sum is exact, so
 * C is the exact product of the dequantised operands up to one rounding per
 * block. qa [M,Kd], sa [M,Kd/128], qb [Nd,Kd] (weights, K contiguous),
 * sb [ceil(Nd/128), Kd/128], C [M,Nd]; all row-major.
 */
void oracle_fp8_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                     int64_t M, int64_t Nd, int64_t Kd, double* C)
{
    tables_init();
    int64_t nkb = Kd / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < nkb; ++kb) {
                double part = 0.0;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    part += g_e4m3_all[qa[m * Kd + k]] * g_e4m3_all[qb[n * Kd + k]];
                acc += (double)sa[m * nkb + kb] * (double)sb[(n / 128) * nkb + kb] * part;
            }
            C[m * Nd + n] = acc;
        }
}

/* C = A B^T for bf16 A [M,Kd] and bf16 B [Nd,Kd]; FP64 sums (products exact). */
void oracle_bf16_gemm(const uint16_t* a, const uint16_t* b, int64_t M, int64_t Nd, int64_t Kd, double* C)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < Kd; ++k)
                acc += oracle_bf16_value(a[m * Kd + k]) * oracle_bf16_value(b[n * Kd + k]);
            C[m * Nd + n] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU expert activation                                                 */
/* ------------------------------------------------------------------------ */

static double silu(double x) { return x / (1.0 + exp(-x)); }

/* a = silu(h1) * h3 in FP64, n elements. */
void oracle_swiglu(const double* h1, const double* h3, int64_t n, double* a)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) a[i] = silu(h1[i]) * h3[i];
}

/*
 * The FP8 path's intermediate: a = silu(h1) * h3 in FP64, rounded once to
 * fp32, then quantised per 1x128 tile as above. rows x I values.
 * dist (optional) gets, per element, the distance of a/scale to the nearest
 * point where its E4M3 code would change (see oracle_e4m3_boundary_distance),
 * and vscaled (optional) the value a/scale itself.
 */
void oracle_swiglu_quant(const double* h1, const double* h3, int64_t rows, int64_t I,
                         uint8_t* q, float* scales, double* dist, double* vscaled)
{
    tables_init();
    int64_t nb = I / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float a32[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) {
                int64_t x = r * I + b * 128 + i;
                a32[i] = (float)(silu(h1[x]) * h3[x]);
            }
            float sc = quant_tile(a32, 128, 1, q + r * I + b * 128, 1);
            scales[r * nb + b] = sc;
            for (int i = 0; i < 128; ++i) {
                float v = a32[i] / sc;
                if (dist) dist[r * I + b * 128 + i] = oracle_e4m3_boundary_distance(v);
                if (vscaled) vscaled[r * I + b * 128 + i] = (double)v;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Combine [formula]                                                        */
/* ------------------------------------------------------------------------ */

/* out[t] = u[t] + y_shared[t] + sum_k g[t,k] * y[dest_row[t,k]] in FP64
 * (y_shared may be NULL: no shared expert). */
void oracle_combine(const uint16_t* u, const uint16_t* y_shared, const uint16_t* y,
                    const double* gates, const int32_t* dest_row,
                    int64_t T, int64_t d, int K, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < d; ++j) {
            double acc = oracle_bf16_value(u[t * d + j]);
            if (y_shared) acc += oracle_bf16_value(y_shared[t * d + j]);
            for (int k = 0; k < K; ++k) {
                int64_t row = dest_row[t * K + k];
                acc += gates[t * K + k] * oracle_bf16_value(y[row * d + j]);
            }
            out[t * d + j] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Bias update [bias]                                                       */
/* ------------------------------------------------------------------------ */

/* With the mean load T*K/N: load above it lowers b_i by gamma, below it
 * raises b_i by gamma, equal leaves it (compared as load*N vs T*K in integers).
 * The update is one fp32 addition. */
void oracle_bias_update(float* bias, const int32_t* loads, int N, int64_t T, int K, float gamma)
{
    int64_t mean_num = T * (int64_t)K;
    for (int i = 0; i < N; ++i) {
        int64_t lhs = (int64_t)loads[i] * N;
        if (lhs > mean_num) bias[i] = bias[i] - gamma;
        else if (lhs < mean_num) bias[i] = bias[i] + gamma;
    }
}

/* ------------------------------------------------------------------------ */
/* Sequence-wise balance statistics [seqloss]                               */
/* ------------------------------------------------------------------------ */

/* Sequences are the consecutive token ranges [s*seq_len, min(T, (s+1)*seq_len)).
 * For sequence s of T_s tokens and expert i:
 *   loads[s][i] = number of (t, k) in the sequence with topk_idx[t,k] == i
 *   prob[s][i]  = (1/T_s) sum_t scores[t,i] / sum_j scores[t,j]
 *   stat[s]     = sum_i (N * loads[s][i] / (K * T_s)) * prob[s][i]
 * scores [T, N] are the affinities s (FP64 here); sums in FP64, in index order. */
void oracle_seq_balance(const double* scores, const int32_t* topk_idx, int64_t T, int N, int K, int64_t seq_len,
                        int32_t* loads, double* prob, double* stat)
{
    const int64_t S = (T + seq_len - 1) / seq_len;
    for (int64_t s = 0; s < S; ++s) {
        const int64_t t0 = s * seq_len, t1 = t0 + seq_len < T ? t0 + seq_len : T;
        const double Ts = (double)(t1 - t0);
        int32_t* ld = loads + s * N;
        double* pr = prob + s * N;
        for (int i = 0; i < N; ++i) {
            ld[i] = 0;
            pr[i] = 0.0;
        }
        for (int64_t t = t0; t < t1; ++t) {
            double row = 0.0;
            for (int i = 0; i < N; ++i) row += scores[t * N + i];
            for (int i = 0; i < N; ++i) pr[i] += scores[t * N + i] / row;
            for (int k = 0; k < K; ++k) ld[topk_idx[t * K + k]] += 1;
        }
        double acc = 0.0;
        for (int i = 0; i < N; ++i) {
            pr[i] /= Ts;
            acc += ((double)N * ld[i] / ((double)K * Ts)) * pr[i];
        }
        stat[s] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Backward pass and training step [train]                                  */
/* ------------------------------------------------------------------------ */

/* Readings (the pages only say that the heavy products of training run in
 * FP8 with the same fine-grained scaling, and that the bias moves after each
 * step): the gradient of the layer formula with the expert choice held fixed
 * and every quantisation or rounding passed straight through; the
 * backward's products use FP8 operands with the [tiles] rule applied along
 * their own contraction dimension, promoted every 128 elements [promote].
 * For a weight gradient the contraction runs over an expert's tokens, so
 * each operand gets one scale per (128 consecutive rows of the expert,
 * column): the activation tile turned on its side. */

/* Quantisation for a weight gradient: x fp32 [R, C] (the rows of one expert),
 * one scale per (block of 128 consecutive rows, column); rows R..Rp-1
 * (Rp = R rounded up to 128) are zeros. q is stored transposed, [C, Rp]
 * (K contiguous, as a product operand), scales [Rp/128, C]. */
void oracle_quant_128x1(const float* x, int64_t R, int64_t C, uint8_t* q, float* scales)
{
    tables_init();
    const int64_t Rp = (R + 127) / 128 * 128, nb = Rp / 128;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        float col[128];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 128; ++i) {
                const int64_t r = b * 128 + i;
                col[i] = r < R ? x[r * C + c] : 0.0f;
            }
            scales[b * C + c] = quant_tile(col, 128, 1, q + c * Rp + b * 128, 1);
        }
    }
}

/* Weight-gradient product: both operands scaled per (128-row block, row):
 *   C[m,n] = sum over blocks b of sa[b,m] * sb[b,n] * sum_{k in b} qa[m,k] * qb[n,k]
 * qa [M, Kp], qb [Nd, Kp] (K contiguous, Kp % 128 == 0), sa [Kp/128, M],
 * sb [Kp/128, Nd]; FP64 block sums (exact), FP64 accumulation in block order. */
void oracle_fp8_gemm_kscaled(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                             int64_t M, int64_t Nd, int64_t Kp, double* C)
{
    tables_init();
    const int64_t nkb = Kp / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            double acc = 0.0;
            for (int64_t b = 0; b < nkb; ++b) {
                double part = 0.0;
                for (int64_t k = b * 128; k < b * 128 + 128; ++k)
                    part += g_e4m3_all[qa[m * Kp + k]] * g_e4m3_all[qb[n * Kp + k]];
                acc += (double)sa[b * M + m] * (double)sb[b * Nd + n] * part;
            }
            C[m * Nd + n] = acc;
        }
}

/* fp32 weights (the training step's master copy): one scale per 128x128
 * block, the [tiles] rule. Layout as oracle_quant_128x128. */
void oracle_quant_128x128_f32(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* scales)
{
    tables_init();
    const int64_t nbr = (rows + 127) / 128, nbc = cols / 128;
#pragma omp parallel for schedule(dynamic)
    for (int64_t br = 0; br < nbr; ++br) {
        const int64_t r0 = br * 128, r1 = r0 + 128 < rows ? r0 + 128 : rows;
        float* buf = (float*)malloc(sizeof(float) * 128 * 128);
        uint8_t* qb = (uint8_t*)malloc(128 * 128);
        for (int64_t bc = 0; bc < nbc; ++bc) {
            int64_t n = 0;
            for (int64_t r = r0; r < r1; ++r)
                for (int i = 0; i < 128; ++i) buf[n++] = w[r * cols + bc * 128 + i];
            scales[br * nbc + bc] = quant_tile(buf, n, 1, qb, 1);
            n = 0;
            for (int64_t r = r0; r < r1; ++r)
                for (int i = 0; i < 128; ++i) q[r * cols + bc * 128 + i] = qb[n++];
        }
        free(buf);
        free(qb);
    }
}

/* SwiGLU backward: with a = silu(h1) * h3 and sig = 1/(1+exp(-h1)),
 *   dh1 = da * h3 * sig * (1 + h1 * (1 - sig)),   dh3 = da * h1 * sig.  FP64. */
void oracle_swiglu_backward(const double* h1, const double* h3, const double* da, int64_t n, double* dh1,
                            double* dh3)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const double sig = 1.0 / (1.0 + exp(-h1[i]));
        dh1[i] = da[i] * h3[i] * sig * (1.0 + h1[i] * (1.0 - sig));
        dh3[i] = da[i] * h1[i] * sig;
    }
}
