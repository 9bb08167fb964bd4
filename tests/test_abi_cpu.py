"""The C library on a machine without a GPU: it loads, exports every entry
point that include/moe.h declares, and rejects bad arguments on the host
(before any CUDA call)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_90_b300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(?:moe_status|size_t|int|const char\*)\s+(\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from mixture_experts_layer_90_b300 import build
    build.build()
    return M.load_library()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(M.EXPORTS) | {"moe_num_sms"}


def test_library_is_sm_103a_only():
    from mixture_experts_layer_90_b300 import build
    assert "arch=compute_103a,code=sm_103a" in build.NVCC_FLAGS


def _ok_ptr():
    return ctypes.c_void_p(4096)


def test_host_validation_rejects_bad_shapes(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    # d not a multiple of 64
    assert L.moe_route(p, 8, 100, p, 1, p, 16, 4, 1, 1, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert b"d=100" in L.moe_last_error()
    # K > 16, N > 1024, groups not dividing N, kept groups too small
    assert L.moe_route(p, 8, 128, p, 1, p, 32, 17, 1, 1, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_route(p, 8, 128, p, 1, p, 2048, 8, 1, 1, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_route(p, 8, 128, p, 1, p, 256, 8, 7, 2, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_route(p, 8, 128, p, 1, p, 256, 8, 64, 1, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    # misaligned token pointer
    assert L.moe_route(ctypes.c_void_p(4098), 8, 128, p, 1, p, 16, 4, 1, 1, p, p, p, None, p, 1 << 20, s) \
        == M.MOE_ERR_INVALID_ARG
    # GEMM shape rules
    assert L.fp8_grouped_gemm(p, p, p, p, p, 4, 100, 384, 256, 0, p, None, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm(p, p, p, p, p, 4, 100, 512, 200, 0, p, None, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm(p, p, p, p, p, 2000, 100, 512, 256, 0, p, None, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm(p, p, p, p, p, 4, 100, 512, 256, 1, p, None, s) == M.MOE_ERR_INVALID_ARG
    assert L.bf16_grouped_gemm(p, p, p, 4, 100, 512, 96, 0, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.bf16_grouped_gemm(p, p, p, 4, 100, 512, 128, 1, p, s) == M.MOE_ERR_INVALID_ARG
    # quantisers
    assert L.fp8_quant_1x128(p, 4, 100, 100, p, p, 4, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_quant_1x128(p, 4, 128, 128, p, p, 3, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_quant_128x128(p, 4, 130, p, p, s) == M.MOE_ERR_INVALID_ARG
    # permute / combine
    assert L.moe_permute(p, 8, 100, p, 16, 4, 0, 0, p, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_permute(p, 8, 128, p, 16, 4, 2, 0, p, p, p, p, None, p, 1 << 20, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_combine(p, None, p, p, p, 8, 100, 4, 40, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_combine(p, None, p, p, p, 8, 128, 0, 40, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_bias_update(None, p, 16, 8, 4, 1e-3, s) == M.MOE_ERR_INVALID_ARG


def test_workspace_rules(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    need = L.moe_route_workspace_size(1000, 1024, 256, M.MOE_DTYPE_F32)
    assert need >= 256 * 3 * 1024 * 2
    assert L.moe_route(p, 1000, 1024, p, 1, p, 256, 8, 1, 1, p, p, p, None, p, need - 1, s) == M.MOE_ERR_WORKSPACE
    assert L.moe_route(p, 1000, 1024, p, 1, p, 256, 8, 1, 1, p, p, p, None, ctypes.c_void_p(4112), need, s) \
        == M.MOE_ERR_WORKSPACE
    assert L.moe_permute_workspace_size(16384, 256) >= 512 * 256 * 4
    w = M.LayerWeights(d=7168, N=256, K=8, I=2048, n_groups=1, topk_groups=1, gamma=1e-3, fp8=1, centroids=8,
                       centroid_dtype=1, bias=8, w13=8, w13_scales=8, w2=8, w2_scales=8)
    n = L.moe_layer_workspace_size(ctypes.byref(w), 8192)
    R = 8192 * 9
    assert n >= R * 7168 * 3 + R * 2048          # x_perm (e4m3) + y (bf16) + intermediate
    assert L.moe_layer_host_workspace_size(ctypes.byref(w), 8192) >= n + 2 * 8192 * 7168 * 2


def test_python_calls_fail_loudly_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError, match="no CUDA device"):
        M.fp8_quant_1x128(torch.zeros((1, 128), dtype=torch.bfloat16))


def _v3_weights():
    p = 4096
    return M.LayerWeights(d=7168, N=256, K=8, I=2048, n_groups=1, topk_groups=1, gamma=1e-3, fp8=1, centroids=p,
                          centroid_dtype=1, bias=p, w13=p, w13_scales=p, w2=p, w2_scales=p)


def test_pipelined_host_call_checks_its_arguments(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    w = _v3_weights()
    outs = M.LayerOutputs(topk_idx=None, gates=None, loads=4096, stage_events=None)
    T = 8192
    need = L.moe_layer_host_pipeline_workspace_size(ctypes.byref(w), T)
    # two device slots for u and for h' on top of the device-buffer workspace
    assert need >= L.moe_layer_workspace_size(ctypes.byref(w), T) + 4 * T * 7168 * 2
    call = lambda slot, ws_bytes, done: L.moe_layer_forward_host_pipelined(  # noqa: E731
        ctypes.byref(w), p, T, p, ctypes.byref(outs), 1, slot, ctypes.c_void_p(1 << 20), ws_bytes, s, done)
    assert call(2, need, p) == M.MOE_ERR_INVALID_ARG
    assert b"slot" in L.moe_last_error()
    assert call(-1, need, p) == M.MOE_ERR_INVALID_ARG
    assert call(0, need, None) == M.MOE_ERR_INVALID_ARG
    assert call(1, need - 1, p) == M.MOE_ERR_WORKSPACE
    no_loads = M.LayerOutputs(topk_idx=None, gates=None, loads=None, stage_events=None)
    assert L.moe_layer_forward_host_pipelined(ctypes.byref(w), p, T, p, ctypes.byref(no_loads), 1, 0,
                                              ctypes.c_void_p(1 << 20), need, s, p) == M.MOE_ERR_INVALID_ARG
    bad = _v3_weights()
    bad.d = 7000
    assert L.moe_layer_forward_host_pipelined(ctypes.byref(bad), p, T, p, ctypes.byref(outs), 1, 0,
                                              ctypes.c_void_p(1 << 20), need, s, p) == M.MOE_ERR_INVALID_ARG


def test_static_permute_checks_its_built_in_scratch_limit(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    call = lambda T, d, N, K, dt=M.MOE_DTYPE_BF16: L.moe_permute_static(  # noqa: E731
        p, T, d, p, N, K, dt, 1, p, p, p, p, p, s)
    # ceil(T/32)*N + N int32 must fit in 2^20: N = 256 allows T <= 131,040; N = 1024 allows T <= 32,736
    assert call(131_072, 128, 256, 8) == M.MOE_ERR_WORKSPACE
    assert b"moe_permute with a workspace" in L.moe_last_error()
    assert call(40_000, 128, 1024, 8) == M.MOE_ERR_WORKSPACE
    # the same argument rules as moe_permute
    assert call(100, 100, 16, 4) == M.MOE_ERR_INVALID_ARG
    assert call(100, 128, 16, 17) == M.MOE_ERR_INVALID_ARG
    assert call(100, 128, 2048, 8) == M.MOE_ERR_INVALID_ARG
    assert call(100, 128, 16, 4, dt=M.MOE_DTYPE_F32) == M.MOE_ERR_INVALID_ARG
    assert L.moe_permute_static(ctypes.c_void_p(4100), 100, 128, p, 16, 4, M.MOE_DTYPE_BF16, 1, p, p, p, p, p,
                                s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_permute_static(p, 100, 128, p, 16, 4, M.MOE_DTYPE_E4M3, 1, p, p, p, p, None,
                                s) == M.MOE_ERR_INVALID_ARG


def test_wait_self_test_limit_is_bounded(L):
    s = ctypes.c_void_p(0)
    assert L.moe_selftest_wait_timeout(0, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_wait_timeout(2_000_000_000, s) == M.MOE_ERR_INVALID_ARG


def test_prepared_routing_checks_its_arguments(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    need = L.moe_route_prepared_centroids_size(7168, 256, M.MOE_DTYPE_F32)
    assert need == 256 * 3 * 7168 * 2                  # three bf16 terms per fp32 centroid value
    assert L.moe_route_prepared_centroids_size(256, 16, M.MOE_DTYPE_BF16) == 256 * 256 * 2   # rows padded to 256
    prep = lambda *a: L.moe_route_prepare_centroids(*a)  # noqa: E731
    assert prep(p, M.MOE_DTYPE_F32, 256, 100, p, need, s) == M.MOE_ERR_INVALID_ARG       # d % 64
    assert prep(p, M.MOE_DTYPE_F32, 2048, 128, p, need, s) == M.MOE_ERR_INVALID_ARG      # N > 1024
    assert prep(p, M.MOE_DTYPE_E4M3, 256, 128, p, need, s) == M.MOE_ERR_INVALID_ARG      # dtype
    assert prep(None, M.MOE_DTYPE_F32, 256, 128, p, need, s) == M.MOE_ERR_INVALID_ARG
    small = L.moe_route_prepared_centroids_size(128, 256, M.MOE_DTYPE_F32)
    assert prep(p, M.MOE_DTYPE_F32, 256, 128, p, small - 1, s) == M.MOE_ERR_WORKSPACE
    assert prep(p, M.MOE_DTYPE_F32, 256, 128, ctypes.c_void_p(4096 + 16), small, s) == M.MOE_ERR_WORKSPACE
    # routing from a prepared operand: the same rules as moe_route, a smaller workspace
    ws = L.moe_route_prepared_workspace_size(1000, 1024, 256, M.MOE_DTYPE_F32)
    assert ws < L.moe_route_workspace_size(1000, 1024, 256, M.MOE_DTYPE_F32)
    call = lambda T, d, N, K, ws_bytes, prepared=p: L.moe_route_prepared(  # noqa: E731
        p, T, d, prepared, M.MOE_DTYPE_F32, p, N, K, 1, 1, p, p, p, None, p, ws_bytes, s)
    assert call(1000, 100, 256, 8, ws) == M.MOE_ERR_INVALID_ARG
    assert call(1000, 1024, 256, 17, ws) == M.MOE_ERR_INVALID_ARG
    assert call(1000, 1024, 256, 8, ws - 1) == M.MOE_ERR_WORKSPACE
    assert call(1000, 1024, 256, 8, ws, prepared=ctypes.c_void_p(4096 + 16)) == M.MOE_ERR_INVALID_ARG
    # a layer given prepared centroids needs no room for them in its workspace
    w = _v3_weights()
    plain = L.moe_layer_workspace_size(ctypes.byref(w), 8192)
    w.centroids_prepared = 4096
    assert L.moe_layer_workspace_size(ctypes.byref(w), 8192) <= plain - 256 * 3 * 7168 * 2


def test_balance_stats_checks_its_arguments(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    call = lambda T, N, K, L_, ws_bytes=1 << 20: L.moe_route_balance_stats(  # noqa: E731
        p, p, T, N, K, L_, p, p, p, p, ws_bytes, s)
    assert call(100, 2048, 8, 10) == M.MOE_ERR_INVALID_ARG
    assert call(100, 64, 17, 10) == M.MOE_ERR_INVALID_ARG
    assert call(100, 4, 8, 10) == M.MOE_ERR_INVALID_ARG        # K > N
    assert call(100, 64, 8, 0) == M.MOE_ERR_INVALID_ARG
    need = L.moe_route_balance_stats_workspace_size(1000, 64, 128)
    assert need >= 8 * 2 * 64 * 8                              # 8 sequences x 2 chunks x 64 experts x 8 bytes
    assert call(1000, 64, 8, 128, need - 1) == M.MOE_ERR_WORKSPACE
    assert call(0, 64, 8, 128, 0) == M.MOE_OK                  # no tokens: nothing to do


def _layer_desc(fp8=1, I=256, d=256, N=8, K=2):
    p = 4096
    return M.LayerWeights(d=d, N=N, K=K, I=I, n_groups=1, topk_groups=1, gamma=1e-3, fp8=fp8, centroids=p,
                          centroid_dtype=M.MOE_DTYPE_F32, bias=p, w13=p, w13_scales=p, w2=p, w2_scales=p,
                          centroids_prepared=None)


def test_training_entry_points_check_their_arguments(L):
    p, s = _ok_ptr(), ctypes.c_void_p(0)
    w = _layer_desc()
    # workspace: the forward's plus H, the affinities and the backward's buffers
    T = 100
    fwd, tr = L.moe_layer_workspace_size(ctypes.byref(w), T), L.moe_layer_train_workspace_size(ctypes.byref(w), T)
    R = T * w.K + T
    assert tr > fwd + R * 2 * w.I * 2 + T * w.N * 4
    # named buffers lie inside the workspace and do not overlap
    spans = []
    for name, which in M.TRAIN_BUFFERS.items():
        off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        assert L.moe_layer_train_buffer(ctypes.byref(w), T, which, ctypes.byref(off), ctypes.byref(nb)) == M.MOE_OK
        assert off.value % 256 == 0 and off.value + nb.value <= tr, name
        spans.append((off.value, off.value + nb.value, name))
    spans.sort()
    for a, b in zip(spans, spans[1:]):
        assert a[1] <= b[0], (a, b)
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.moe_layer_train_buffer(ctypes.byref(w), T, 99, ctypes.byref(off), ctypes.byref(nb)) \
        == M.MOE_ERR_INVALID_ARG
    # bf16 layers and I not a multiple of 256 are refused
    outs = M.LayerOutputs(topk_idx=None, gates=None, loads=4096, stage_events=None)
    wb = _layer_desc(fp8=0)
    assert L.moe_layer_forward_train(ctypes.byref(wb), p, T, p, ctypes.byref(outs), 1, p, 1 << 40, s) \
        == M.MOE_ERR_UNSUPPORTED
    wi = _layer_desc(I=384)
    assert L.moe_layer_forward_train(ctypes.byref(wi), p, T, p, ctypes.byref(outs), 1, p, 1 << 40, s) \
        == M.MOE_ERR_INVALID_ARG
    # a dispatch mode that does not exist
    wd = _layer_desc()
    wd.dispatch = 7
    assert L.moe_layer_forward(ctypes.byref(wd), p, T, p, ctypes.byref(outs), 1, p, 1 << 40, s) \
        == M.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward_train(ctypes.byref(wd), p, T, p, ctypes.byref(outs), 1, p, 1 << 40, s) \
        == M.MOE_ERR_INVALID_ARG
    # a too-small workspace
    assert L.moe_layer_forward_train(ctypes.byref(w), p, T, p, ctypes.byref(outs), 1, p, tr - 1, s) \
        == M.MOE_ERR_WORKSPACE
    # the backward needs the transposed weights and every gradient buffer
    wt = M.LayerWeightsT(w13t=4096, w13t_scales=4096, w2t=4096, w2t_scales=4096)
    g_missing = M.LayerGrads(dw13=4096, dw2=None, dcentroids=4096, dz=None, stage_events=None)
    assert L.moe_layer_backward(ctypes.byref(w), ctypes.byref(wt), p, T, p, p, ctypes.byref(g_missing), p, tr, s) \
        == M.MOE_ERR_INVALID_ARG
    wt0 = M.LayerWeightsT(w13t=None, w13t_scales=4096, w2t=4096, w2t_scales=4096)
    g = M.LayerGrads(dw13=4096, dw2=4096, dcentroids=4096, dz=None, stage_events=None)
    assert L.moe_layer_backward(ctypes.byref(w), ctypes.byref(wt0), p, T, p, p, ctypes.byref(g), p, tr, s) \
        == M.MOE_ERR_INVALID_ARG
    # the training step needs fp32 centroids and masters
    m = M.LayerMasters(w13=None, w2=4096)
    assert L.moe_layer_train_step(ctypes.byref(w), ctypes.byref(wt), ctypes.byref(m), p, T, p, 0.1, p, p,
                                  ctypes.byref(outs), ctypes.byref(g), p, tr, s) == M.MOE_ERR_INVALID_ARG
    wc = _layer_desc()
    wc.centroid_dtype = M.MOE_DTYPE_BF16
    m = M.LayerMasters(w13=4096, w2=4096)
    assert L.moe_layer_train_step(ctypes.byref(wc), ctypes.byref(wt), ctypes.byref(m), p, T, p, 0.1, p, p,
                                  ctypes.byref(outs), ctypes.byref(g), p, tr, s) == M.MOE_ERR_UNSUPPORTED
    # weight-gradient GEMM, transpose and SGD shape rules
    assert L.fp8_grouped_gemm_wgrad(p, p, p, p, p, 4, 100, 256, 256, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm_wgrad(p, p, p, p, p, 4, 128, 128, 256, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm_wgrad(p, p, p, p, p, 4, 128, 256, 200, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_grouped_gemm_wgrad(p, p, p, p, p, 2000, 128, 256, 256, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.fp8_transpose_128x128(p, p, 1, 100, 128, p, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_sgd_requant_128x128(p, p, 1, 128, 96, 0.1, p, p, p, p, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_sgd_f32(p, p, -1, 0.1, s) == M.MOE_ERR_INVALID_ARG
    assert L.moe_sgd_f32(None, None, 0, 0.1, s) == M.MOE_OK
