"""moe_permute_static: the permutation for callers that cannot allocate device
memory (no workspace argument; its scratch is a fixed array inside the
library). Through the C ABI it must give exactly what moe_permute gives with a
caller workspace, on consecutive calls that share the library's scratch.

Kept in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


def _lib():
    import mixture_experts_layer_90_b300 as m
    return m


def _topk(T, N, K, seed):
    h = S.bits(S.key(seed, "static-topk", T, N, K), 0, T * N).view(T, N)
    return torch.sort(torch.argsort(h, dim=1)[:, :K], dim=1).values.to(torch.int32)


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return torch.equal(a, b)


@pytest.mark.parametrize("cases", [
    # two calls in a row: different sizes, so stale scratch from the first would show in the second
    [(1000, 512, 64, 6, False, True), (333, 640, 256, 8, True, True)],
    [(4096, 256, 256, 8, True, False), (17, 128, 16, 4, False, False)],
])
def test_static_scratch_matches_workspace_path(cases):
    m = _lib()
    for T, d, N, K, fp8, shared in cases:
        x = S.normal((T, d), 1.0, S.key(0, "static-x", T, d)).cuda()
        idx = _topk(T, N, K, seed=T).cuda()
        dt = m.MOE_DTYPE_E4M3 if fp8 else m.MOE_DTYPE_BF16
        got = m.moe_permute_static(x, idx, N, dt, with_shared=shared)
        exp = m.moe_permute(x, idx, N, dt, with_shared=shared)
        assert m.device_status() == 0
        for g, e in zip(got, exp):
            assert _same(g, e)


def test_static_scratch_rejects_sizes_beyond_its_limit():
    m = _lib()
    L = m.load_library()
    p = ctypes.c_void_p(4096)
    # ceil(T/32)*N + N > 2^20 int32: T = 131072, N = 256 -> 4096*256 + 256
    st = L.moe_permute_static(p, 131072, 128, p, 256, 8, m.MOE_DTYPE_BF16, 0, p, p, p, p, None,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MOE_ERR_WORKSPACE
    assert b"built-in scratch" in L.moe_last_error()
