// The C ABI of training (include/moe.h, "Training"): the training forward,
// the backward pass, one SGD step, and their workspace. Part of the library's
// single translation unit, after abi.cu (whose validation helpers, workspace
// layout and layer forward it uses).

namespace {

// The training workspace: the forward's (LayerWs), then the buffers below.
struct TrainWs {
    LayerWs fwd;
    size_t H, scores, logits, row_gate, dg, qdy, sdy, dA, dH, qdh, sdh, dX, kofs, dz_row, prow;
    size_t qyt, syt, qat, sat, qht, sht, qxt, sxt;
    int64_t Kp;   // padded token rows of the weight-gradient operands
    size_t total;
};

TrainWs train_ws(const moe_layer_weights* w, int64_t T) {
    TrainWs W{};
    W.fwd = layer_ws(w, T, 0);
    const int64_t R = T * w->K + T;
    const int G = w->N + 1;
    const size_t d = size_t(w->d), I = size_t(w->I);
    // every group adds at most one partial block of 128 rows
    W.Kp = ((R + 127) / 128 + G) * 128;
    size_t o = W.fwd.total;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += up256(bytes);
        return at;
    };
    W.H = take(size_t(R) * 2 * I * 2);
    W.scores = take(size_t(T) * w->N * 4);
    W.logits = take(size_t(T) * w->N * 4);
    W.row_gate = take(size_t(R) * 4);
    W.dg = take(size_t(T) * w->K * 4);
    W.qdy = take(size_t(R) * d);
    W.sdy = take(d / 128 * size_t(R) * 4);
    W.dA = take(size_t(R) * I * 2);
    W.dH = take(size_t(R) * 2 * I * 2);
    W.qdh = take(size_t(R) * 2 * I);
    W.sdh = take(2 * I / 128 * size_t(R) * 4);
    W.dX = take(size_t(R) * d * 2);
    W.kofs = take(size_t(G + 1) * 4);
    W.dz_row = take(size_t(T) * w->K * 4);
    const size_t Kp = size_t(W.Kp), nkb = Kp / 128;
    W.prow = take(Kp * 4);
    W.qyt = take(d * Kp);
    W.syt = take(nkb * d * 4);
    W.qat = take(I * Kp);
    W.sat = take(nkb * I * 4);
    W.qht = take(2 * I * Kp);
    W.sht = take(nkb * 2 * I * 4);
    W.qxt = take(d * Kp);
    W.sxt = take(nkb * d * 4);
    W.total = o;
    return W;
}

moe_status check_train(const moe_layer_weights* w, const char* who) {
    STATUS_OK(check_layer(w));
    UNSUPPORTED(w->fp8, "%s: training needs a FP8 layer", who);
    REQUIRE(w->I % 256 == 0, "%s: I=%d must be a multiple of 256", who, w->I);
    return MOE_OK;
}

moe_status check_ws(void* ws, size_t bytes, size_t need, const char* who) {
    if (!ws || bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(MOE_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-byte aligned", who, need);
    return MOE_OK;
}

moe_status wgrad_gemm(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb, const int32_t* kofs,
                      int G, int M, int Nd, int64_t Kp, float* C, moe_stream_t stream) {
    CUtensorMap ta, tb, tc;
    if (!moe::make_kmajor_map(&ta, A, false, uint64_t(Kp), uint64_t(M), uint64_t(Kp), 128) ||
        !moe::make_kmajor_map(&tb, B, false, uint64_t(Kp), uint64_t(Nd), uint64_t(Kp), 256) ||
        !moe::make_f32_store_map(&tc, C, uint64_t(Nd), uint64_t(G) * M))
        return fail(MOE_ERR_CUDA, "fp8_grouped_gemm_wgrad: tensor map encoding failed");
    moe::GemmArgs a{};
    a.group_offsets = kofs;
    a.G = G;
    a.M_total = M;
    a.Nd = Nd;
    a.Kd = int(Kp);
    a.k_steps = int(Kp / 128);
    a.a_k_repeat = 1;
    a.elems_per_step = 128;
    a.splits = 1;
    a.epilogue = MOE_EPI_F32;
    a.sa = sa;
    a.lda_s = M;
    a.sb = sb;
    a.C = C;
    CUDA_OK(moe::run_grouped_gemm(moe::kModeFP8W, ta, tb, a, moe::num_sms(), stream, &tc));
    return MOE_OK;
}

moe_status layer_backward(const moe_layer_weights* w, const moe_layer_weights_t* wt, const uint16_t* u, int64_t T,
                          const uint16_t* dout, uint16_t* du, const moe_layer_grads* gr, uint8_t* ws,
                          const TrainWs& W, moe_stream_t stream) {
    const int K = w->K, N = w->N, d = w->d, I = w->I, G = N + 1;
    const int64_t R = T * K + T;
    if (T == 0) {
        if (gr->stage_events)
            for (int i = 0; i <= MOE_BACKWARD_STAGES; ++i)
                CUDA_OK(cudaEventRecord(reinterpret_cast<cudaEvent_t>(gr->stage_events[i]), stream));
        // no token: every gradient is zero
        CUDA_OK(cudaMemsetAsync(gr->dw13, 0, size_t(G) * 2 * I * d * 4, stream));
        CUDA_OK(cudaMemsetAsync(gr->dw2, 0, size_t(G) * d * I * 4, stream));
        CUDA_OK(cudaMemsetAsync(gr->dcentroids, 0, size_t(N) * d * 4, stream));
        return MOE_OK;
    }
    const LayerWs& L = W.fwd;
    const int32_t* offsets = reinterpret_cast<const int32_t*>(ws + L.offsets);
    const int32_t* perm_token = reinterpret_cast<const int32_t*>(ws + L.perm_token);
    const int32_t* dest = reinterpret_cast<const int32_t*>(ws + L.dest_row);
    const int32_t* topk = reinterpret_cast<const int32_t*>(ws + L.topk);
    const float* gates = reinterpret_cast<const float*>(ws + L.gates);
    const uint16_t* y = reinterpret_cast<const uint16_t*>(ws + L.y);
    const uint16_t* H = reinterpret_cast<const uint16_t*>(ws + W.H);
    const float* scores = reinterpret_cast<const float*>(ws + W.scores);
    const float* logits = reinterpret_cast<const float*>(ws + W.logits);
    float* row_gate = reinterpret_cast<float*>(ws + W.row_gate);
    float* dg = reinterpret_cast<float*>(ws + W.dg);
    uint8_t* qdy = ws + W.qdy;
    float* sdy = reinterpret_cast<float*>(ws + W.sdy);
    uint16_t* dA = reinterpret_cast<uint16_t*>(ws + W.dA);
    uint16_t* dH = reinterpret_cast<uint16_t*>(ws + W.dH);
    uint8_t* qdh = ws + W.qdh;
    float* sdh = reinterpret_cast<float*>(ws + W.sdh);
    uint16_t* dX = reinterpret_cast<uint16_t*>(ws + W.dX);
    int32_t* kofs = reinterpret_cast<int32_t*>(ws + W.kofs);
    float* dz_row = reinterpret_cast<float*>(ws + W.dz_row);
    auto mark = [&](int i) -> moe_status {
        if (gr->stage_events) CUDA_OK(cudaEventRecord(reinterpret_cast<cudaEvent_t>(gr->stage_events[i]), stream));
        return MOE_OK;
    };

    STATUS_OK(mark(0));
    // combine backward: dg and the dgrad operand dY (1x128 tiles)
    CUDA_OK(moe::launch_combine_bwd(dout, y, gates, dest, T, d, K, R, qdy, sdy, row_gate, dg, stream));
    STATUS_OK(mark(1));
    // dA = dY W2 (W2's blocks transposed), bf16
    STATUS_OK(fp8_gemm_impl(qdy, sdy, wt->w2t, wt->w2t_scales, offsets, G, R, I, d, MOE_EPI_BF16, dA, nullptr,
                            nullptr, stream));
    STATUS_OK(mark(2));
    // dH from H and dA, bf16 and 1x128 tiles
    CUDA_OK(moe::launch_swiglu_bwd(dA, H, R, I, dH, qdh, sdh, stream));
    STATUS_OK(mark(3));
    // dX = dH W13 (W13's blocks transposed), bf16
    STATUS_OK(fp8_gemm_impl(qdh, sdh, wt->w13t, wt->w13t_scales, offsets, G, R, d, 2 * I, MOE_EPI_BF16, dX,
                            nullptr, nullptr, stream));
    STATUS_OK(mark(4));
    // gates and du
    CUDA_OK(moe::launch_unpermute_bwd(dout, dX, dest, topk, gates, scores, logits, dg, w->centroids,
                                      w->centroid_dtype == MOE_DTYPE_F32, T, d, N, K, du, dz_row, gr->dz, stream));
    CUDA_OK(moe::launch_centroid_grad(u, offsets, perm_token, dz_row, N, d, gr->dcentroids, stream));
    STATUS_OK(mark(5));
    // weight gradients: operands per (128 tokens of an expert, column), transposed
    CUDA_OK(moe::launch_kblock_offsets(offsets, G, kofs, stream));
    const int64_t Kp = W.Kp, TK = T * K;
    int32_t* prow = reinterpret_cast<int32_t*>(ws + W.prow);
    CUDA_OK(moe::launch_pad_rows(offsets, kofs, G, Kp, prow, stream));
    uint8_t* qyt = ws + W.qyt;
    uint8_t* qat = ws + W.qat;
    uint8_t* qht = ws + W.qht;
    uint8_t* qxt = ws + W.qxt;
    float* syt = reinterpret_cast<float*>(ws + W.syt);
    float* sat = reinterpret_cast<float*>(ws + W.sat);
    float* sht = reinterpret_cast<float*>(ws + W.sht);
    float* sxt = reinterpret_cast<float*>(ws + W.sxt);
    CUDA_OK(moe::launch_quant_t(moe::kQuantTScaledG, prow, kofs, G, TK, perm_token, row_gate, dout, d, Kp, qyt,
                                syt, stream));
    CUDA_OK(moe::launch_quant_t(moe::kQuantTSwiglu, prow, kofs, G, TK, perm_token, nullptr, H, I, Kp, qat, sat,
                                stream));
    CUDA_OK(moe::launch_quant_t(moe::kQuantTRows, prow, kofs, G, TK, perm_token, nullptr, dH, 2 * I, Kp, qht, sht,
                                stream));
    CUDA_OK(moe::launch_quant_t(moe::kQuantTTokens, prow, kofs, G, TK, perm_token, nullptr, u, d, Kp, qxt, sxt,
                                stream));
    STATUS_OK(mark(6));
    // dW2 = dY^T A  [G][d][I];  dW13 = dH^T X  [G][2I][d]
    STATUS_OK(wgrad_gemm(qyt, syt, qat, sat, kofs, G, d, I, Kp, gr->dw2, stream));
    STATUS_OK(mark(7));
    STATUS_OK(wgrad_gemm(qht, sht, qxt, sxt, kofs, G, 2 * I, d, Kp, gr->dw13, stream));
    STATUS_OK(mark(8));
    return MOE_OK;
}

moe_status check_backward_args(const moe_layer_weights* w, const moe_layer_weights_t* wt, const uint16_t* u,
                               int64_t T, const uint16_t* dout, const uint16_t* du, const moe_layer_grads* gr,
                               const char* who) {
    STATUS_OK(check_train(w, who));
    REQUIRE(T >= 0 && T * (w->K + 1) <= kMaxRows, "%s: T=%lld out of range", who, (long long)T);
    REQUIRE(wt && wt->w13t && wt->w13t_scales && wt->w2t && wt->w2t_scales, "%s: null transposed weights", who);
    REQUIRE(gr && gr->dw13 && gr->dw2 && gr->dcentroids, "%s: null gradient buffer", who);
    REQUIRE(al16(wt->w13t) && al16(wt->w2t) && al32(gr->dw13) && al32(gr->dw2) && al16(gr->dcentroids) &&
                al16(w->centroids),
            "%s: misaligned weight, centroid or gradient buffer", who);
    if (T > 0) {
        REQUIRE(u && dout && du, "%s: null u/dout/du", who);
        REQUIRE(al16(u) && al16(dout) && al16(du), "%s: u, dout and du must be 16-byte aligned", who);
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_layer_train_workspace_size(const moe_layer_weights* w, int64_t T) { return w ? train_ws(w, T).total : 0; }

moe_status moe_layer_train_buffer(const moe_layer_weights* w, int64_t T, int which, size_t* offset, size_t* bytes) {
    REQUIRE(w && offset && bytes && T >= 0, "moe_layer_train_buffer: bad arguments");
    const TrainWs W = train_ws(w, T);
    const int64_t R = T * w->K + T;
    const size_t d = size_t(w->d), I = size_t(w->I);
    switch (which) {
        case MOE_TRAIN_H: *offset = W.H; *bytes = size_t(R) * 2 * I * 2; break;
        case MOE_TRAIN_SCORES: *offset = W.scores; *bytes = size_t(T) * w->N * 4; break;
        case MOE_TRAIN_DG: *offset = W.dg; *bytes = size_t(T) * w->K * 4; break;
        case MOE_TRAIN_DA: *offset = W.dA; *bytes = size_t(R) * I * 2; break;
        case MOE_TRAIN_DH: *offset = W.dH; *bytes = size_t(R) * 2 * I * 2; break;
        case MOE_TRAIN_DX: *offset = W.dX; *bytes = size_t(R) * d * 2; break;
        case MOE_TRAIN_OFFSETS: *offset = W.fwd.offsets; *bytes = size_t(w->N + 2) * 4; break;
        case MOE_TRAIN_PERM_TOKEN: *offset = W.fwd.perm_token; *bytes = size_t(T) * w->K * 4; break;
        case MOE_TRAIN_DEST_ROW: *offset = W.fwd.dest_row; *bytes = size_t(T) * w->K * 4; break;
        case MOE_TRAIN_Y: *offset = W.fwd.y; *bytes = size_t(R) * d * 2; break;
        case MOE_TRAIN_KOFS: *offset = W.kofs; *bytes = size_t(w->N + 2) * 4; break;
        case MOE_TRAIN_DY_Q: *offset = W.qdy; *bytes = size_t(R) * d; break;
        case MOE_TRAIN_DY_S: *offset = W.sdy; *bytes = d / 128 * size_t(R) * 4; break;
        case MOE_TRAIN_DH_Q: *offset = W.qdh; *bytes = size_t(R) * 2 * I; break;
        case MOE_TRAIN_DH_S: *offset = W.sdh; *bytes = 2 * I / 128 * size_t(R) * 4; break;
        case MOE_TRAIN_ROW_GATE: *offset = W.row_gate; *bytes = size_t(R) * 4; break;
        case MOE_TRAIN_LOGITS: *offset = W.logits; *bytes = size_t(T) * w->N * 4; break;
        default: return fail(MOE_ERR_INVALID_ARG, "moe_layer_train_buffer: unknown buffer %d", which);
    }
    return MOE_OK;
}

moe_status moe_layer_forward_train(const moe_layer_weights* w, const uint16_t* u, int64_t T, uint16_t* out,
                                   const moe_layer_outputs* outs, int update_bias, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream) {
    STATUS_OK(check_train(w, "moe_layer_forward_train"));
    REQUIRE(outs && outs->loads, "moe_layer_forward_train: outputs need a loads buffer");
    REQUIRE(T >= 0 && T * (w->K + 1) <= kMaxRows && (T == 0 || (u && out)), "moe_layer_forward_train: bad u/out/T");
    const TrainWs W = train_ws(w, T);
    STATUS_OK(check_ws(workspace, workspace_bytes, W.total, "moe_layer_forward_train"));
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    // the routing and the gates stay in the workspace for the backward
    moe_layer_outputs o = *outs;
    o.topk_idx = nullptr;
    o.gates = nullptr;
    STATUS_OK(layer_forward(w, u, T, out, &o, update_bias, ws, W.fwd, stream, reinterpret_cast<float*>(ws + W.scores),
                            reinterpret_cast<uint16_t*>(ws + W.H), reinterpret_cast<float*>(ws + W.logits)));
    const size_t tk = size_t(T) * w->K;
    if (T > 0 && outs->topk_idx)
        CUDA_OK(cudaMemcpyAsync(outs->topk_idx, ws + W.fwd.topk, tk * 4, cudaMemcpyDeviceToDevice, stream));
    if (T > 0 && outs->gates)
        CUDA_OK(cudaMemcpyAsync(outs->gates, ws + W.fwd.gates, tk * 4, cudaMemcpyDeviceToDevice, stream));
    return MOE_OK;
}

moe_status moe_layer_backward(const moe_layer_weights* w, const moe_layer_weights_t* wt, const uint16_t* u,
                              int64_t T, const uint16_t* dout, uint16_t* du, const moe_layer_grads* grads,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    STATUS_OK(check_backward_args(w, wt, u, T, dout, du, grads, "moe_layer_backward"));
    const TrainWs W = train_ws(w, T);
    STATUS_OK(check_ws(workspace, workspace_bytes, W.total, "moe_layer_backward"));
    return layer_backward(w, wt, u, T, dout, du, grads, reinterpret_cast<uint8_t*>(workspace), W, stream);
}

moe_status fp8_grouped_gemm_wgrad(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                                  const int32_t* kofs, int G, int M, int Nd, int64_t Kp, float* C,
                                  moe_stream_t stream) {
    REQUIRE(G >= 1 && G <= moe::gemm_max_groups(), "fp8_grouped_gemm_wgrad: G=%d must be in [1, 1024]", G);
    REQUIRE(M > 0 && M % 128 == 0, "fp8_grouped_gemm_wgrad: M=%d must be a positive multiple of 128", M);
    REQUIRE(Nd > 0 && Nd % 256 == 0, "fp8_grouped_gemm_wgrad: Nd=%d must be a positive multiple of 256", Nd);
    REQUIRE(Kp > 0 && Kp % 128 == 0 && Kp <= kMaxRows, "fp8_grouped_gemm_wgrad: Kp must be a multiple of 128");
    REQUIRE(int64_t(G) * M <= kMaxRows, "fp8_grouped_gemm_wgrad: G*M too large");
    REQUIRE(A && sa && B && sb && kofs && C, "fp8_grouped_gemm_wgrad: null pointer");
    REQUIRE(al16(A) && al16(B) && al16(sa) && al16(sb) && al32(C), "fp8_grouped_gemm_wgrad: misaligned pointer");
    return wgrad_gemm(A, sa, B, sb, kofs, G, M, Nd, Kp, C, stream);
}

moe_status fp8_transpose_128x128(const uint8_t* q, const float* s, int G, int rows, int cols, uint8_t* qt,
                                 float* st, moe_stream_t stream) {
    REQUIRE(G >= 1 && G <= 65535, "fp8_transpose_128x128: G=%d", G);
    REQUIRE(rows > 0 && rows % 128 == 0 && cols > 0 && cols % 128 == 0 && rows / 128 <= 65535,
            "fp8_transpose_128x128: rows and cols must be positive multiples of 128");
    REQUIRE(q && s && qt && st, "fp8_transpose_128x128: null pointer");
    REQUIRE(al16(q) && al16(qt), "fp8_transpose_128x128: q and qt must be 16-byte aligned");
    CUDA_OK(moe::launch_fp8_transpose(q, s, G, rows, cols, qt, st, stream));
    return MOE_OK;
}

moe_status moe_sgd_requant_128x128(float* w, const float* grad, int G, int rows, int cols, float lr, uint8_t* q,
                                   float* s, uint8_t* qt, float* st, moe_stream_t stream) {
    REQUIRE(G >= 1 && G <= 65535, "moe_sgd_requant_128x128: G=%d", G);
    REQUIRE(rows > 0 && rows % 128 == 0 && cols > 0 && cols % 128 == 0 && rows / 128 <= 65535,
            "moe_sgd_requant_128x128: rows and cols must be positive multiples of 128");
    REQUIRE(w && grad && q && s && qt && st, "moe_sgd_requant_128x128: null pointer");
    REQUIRE(al16(w) && al16(grad) && al16(q) && al16(qt), "moe_sgd_requant_128x128: misaligned pointer");
    CUDA_OK(moe::launch_sgd_requant(w, grad, G, rows, cols, lr, q, s, qt, st, stream));
    return MOE_OK;
}

moe_status moe_sgd_f32(float* w, const float* grad, int64_t n, float lr, moe_stream_t stream) {
    REQUIRE(n >= 0, "moe_sgd_f32: n < 0");
    if (n == 0) return MOE_OK;
    REQUIRE(w && grad, "moe_sgd_f32: null pointer");
    CUDA_OK(moe::launch_sgd_f32(w, grad, n, lr, stream));
    return MOE_OK;
}

moe_status moe_layer_train_step(const moe_layer_weights* w, const moe_layer_weights_t* wt,
                                const moe_layer_masters* m, const uint16_t* u, int64_t T, const uint16_t* dout,
                                float lr, uint16_t* out, uint16_t* du, const moe_layer_outputs* outs,
                                const moe_layer_grads* grads, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
    STATUS_OK(check_backward_args(w, wt, u, T, dout, du, grads, "moe_layer_train_step"));
    REQUIRE(m && m->w13 && m->w2 && al16(m->w13) && al16(m->w2), "moe_layer_train_step: bad master weights");
    UNSUPPORTED(w->centroid_dtype == MOE_DTYPE_F32, "moe_layer_train_step: the centroids must be fp32");
    STATUS_OK(moe_layer_forward_train(w, u, T, out, outs, 1, workspace, workspace_bytes, stream));
    STATUS_OK(moe_layer_backward(w, wt, u, T, dout, du, grads, workspace, workspace_bytes, stream));
    const int G = w->N + 1, d = w->d, I = w->I;
    STATUS_OK(moe_sgd_requant_128x128(m->w13, grads->dw13, G, 2 * I, d, lr,
                                      static_cast<uint8_t*>(const_cast<void*>(w->w13)),
                                      const_cast<float*>(w->w13_scales), wt->w13t, wt->w13t_scales, stream));
    STATUS_OK(moe_sgd_requant_128x128(m->w2, grads->dw2, G, d, I, lr, static_cast<uint8_t*>(const_cast<void*>(w->w2)),
                                      const_cast<float*>(w->w2_scales), wt->w2t, wt->w2t_scales, stream));
    STATUS_OK(moe_sgd_f32(static_cast<float*>(const_cast<void*>(w->centroids)), grads->dcentroids,
                          int64_t(w->N) * d, lr, stream));
    if (w->centroids_prepared) {
        const size_t pb = moe::prepared_centroid_bytes(d, w->N, w->centroid_dtype);
        STATUS_OK(moe_route_prepare_centroids(w->centroids, w->centroid_dtype, w->N, d,
                                              const_cast<void*>(w->centroids_prepared), pb, stream));
    }
    return MOE_OK;
}

}  // extern "C"
