"""Edge cases of the entry points on the GPU: empty inputs, the largest group
count the grouped GEMM accepts, and the degenerate cases of the routing rule
(every expert chosen; group limits that keep every group)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import ROUTE_DELTA, check_bf16

pytestmark = pytest.mark.gpu


def _lib():
    import mixture_experts_layer_90_b300 as m
    return m


def test_empty_inputs_do_nothing_and_report_nothing():
    m = _lib()
    d, N, K = 256, 16, 4
    x = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    q, s = m.fp8_quant_1x128(x)
    assert q.shape == (0, d)
    cent = S.centroids(S.LayerShape(T=0, d=d, N=N, K=K, I=128)).cuda()
    bias = torch.zeros(N, device="cuda")
    idx, gates, loads, _ = m.moe_route(x, cent, bias, K)
    assert idx.shape == (0, K) and int(loads.abs().sum()) == 0
    off, perm, dest, xp, xs = m.moe_permute(x, idx, N, m.MOE_DTYPE_E4M3, with_shared=True)
    assert (off.cpu() == 0).all()
    A = torch.empty((0, d), dtype=torch.uint8, device="cuda")
    sa = torch.empty((d // 128, 0), dtype=torch.float32, device="cuda")
    B = torch.zeros((2, 256, d), dtype=torch.uint8, device="cuda")
    sb = torch.ones((2, 2, d // 128), dtype=torch.float32, device="cuda")
    C = m.fp8_grouped_gemm(A, sa, B, sb, torch.zeros(3, dtype=torch.int32, device="cuda"))
    assert C.shape == (0, 256)
    out = m.moe_combine(x, None, torch.empty((0, d), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((0, K), device="cuda"), torch.empty((0, K), dtype=torch.int32, device="cuda"))
    assert out.shape == (0, d)
    assert m.device_status() == m.MOE_OK


def test_grouped_gemm_with_the_largest_group_count():
    """1024 groups, most of them empty, a few ragged ones, rows of the last group at the end."""
    m = _lib()
    G, Nd, Kd = 1024, 256, 256
    sizes = np.zeros(G, np.int64)
    sizes[[0, 5, 511, 1000, 1023]] = [3, 130, 1, 77, 128]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1])
    a = S.normal((M, Kd), 1.0, S.key(0, "g1024-a"))
    qa, sa = oracle.quant_1x128(a)
    live = np.nonzero(sizes)[0]
    qb = np.zeros((G, Nd, Kd), np.uint8)
    sb = np.ones((G, Nd // 128, Kd // 128), np.float32)
    for g in live:
        w = S.normal((Nd, Kd), 0.05, S.key(0, "g1024-b", int(g)))
        qb[g], sb[g] = oracle.quant_128x128(w)
    C = m.fp8_grouped_gemm(torch.as_tensor(qa).cuda(), torch.as_tensor(np.ascontiguousarray(sa.T)).cuda(),
                           torch.as_tensor(qb).cuda(), torch.as_tensor(sb).cuda(), torch.as_tensor(offs).cuda())
    assert m.device_status() == m.MOE_OK
    C = C.cpu()
    for g in live:
        r0, r1 = offs[g], offs[g + 1]
        check_bf16(C[r0:r1], oracle.fp8_gemm(qa[r0:r1], sa[r0:r1], qb[g], sb[g]), what=f"group {g}")


def test_route_every_expert_chosen():
    """K = N: every expert is chosen, the gates are s / sum(s) over all experts."""
    m = _lib()
    T, d, N = 64, 512, 16
    u = S.normal((T, d), 1.0, S.key(0, "kn-u"))
    e = S.normal((N, d), 1.0 / math.sqrt(d), S.key(0, "kn-e"), dtype=torch.float32)
    b = S.uniform((N,), -0.01, 0.01, S.key(0, "kn-b"))
    idx, gates, loads, scores = m.moe_route(u.cuda(), e.cuda(), b.cuda(), N, want_scores=True)
    assert m.device_status() == m.MOE_OK
    assert (idx.cpu() == torch.arange(N, dtype=torch.int32)).all()
    assert (loads.cpu() == T).all()
    s = scores.cpu().double()
    np.testing.assert_allclose(gates.cpu().double().numpy(), (s / s.sum(1, keepdim=True)).numpy(), rtol=3e-6)


def test_group_limit_keeping_every_group_is_flat_routing():
    m = _lib()
    T, d, N, K = 200, 512, 64, 6
    u = S.normal((T, d), 1.0, S.key(0, "gl-u"))
    e = S.normal((N, d), 1.0 / math.sqrt(d), S.key(0, "gl-e"), dtype=torch.float32)
    b = S.uniform((N,), -0.01, 0.01, S.key(0, "gl-b"))
    flat = m.moe_route(u.cuda(), e.cuda(), b.cuda(), K)
    grouped = m.moe_route(u.cuda(), e.cuda(), b.cuda(), K, n_groups=8, topk_groups=8)
    assert m.device_status() == m.MOE_OK
    assert torch.equal(flat[0], grouped[0]) and torch.equal(flat[2], grouped[2])
    assert torch.equal(flat[1], grouped[1])
