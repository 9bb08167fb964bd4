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
