"""Device-side failure detection, tested without faulting the GPU.

Each case makes a kernel meet a problem that its own checks turn into a
device status (read and cleared by moe_get_device_status), after which the
context must still run ordinary calls:
  * a bounded wait on an mbarrier that nothing arrives on times out;
  * expert ids outside [0, N) reach the permutation;
  * group offsets that decrease reach the grouped GEMM;
  * a destination row outside [0, R) reaches the combine.
"""
import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


def _lib():
    import mixture_experts_layer_90_b300 as m
    return m


def _context_still_works():
    m = _lib()
    x = S.normal((64, 256), 1.0, S.key(0, "err-after")).cuda()
    q, s = m.fp8_quant_1x128(x)
    assert m.device_status() == m.MOE_OK
    assert q.shape == (64, 256)


def test_bounded_wait_times_out_and_reports():
    m = _lib()
    m.moe_selftest_wait_timeout(2_000_000)            # 2 ms
    assert m.device_status() == m.MOE_ERR_TIMEOUT
    assert m.device_status() == m.MOE_OK              # reading clears the word
    _context_still_works()


def test_permute_reports_out_of_range_expert_ids():
    m = _lib()
    T, d, N, K = 100, 256, 16, 4
    x = S.normal((T, d), 1.0, S.key(0, "err-perm")).cuda()
    idx = torch.arange(K, dtype=torch.int32).repeat(T, 1)
    idx[3, 1] = N            # one id past the last expert
    idx[50, 0] = -3          # one negative id
    for out_dtype in (m.MOE_DTYPE_BF16, m.MOE_DTYPE_E4M3):
        off, perm, dest, xp, xs = m.moe_permute(x, idx.cuda(), N, out_dtype, with_shared=True)
        assert m.device_status() == m.MOE_ERR_DEVICE_DATA
        dest = dest.cpu().numpy()
        assert dest[3, 1] == -1 and dest[50, 0] == -1
        # the valid pairs still got their rows
        assert (np.delete(dest.ravel(), [3 * K + 1, 50 * K]) >= 0).all()
    _context_still_works()


def test_grouped_gemm_reports_decreasing_offsets():
    m = _lib()
    G, Nd, Kd, M = 3, 256, 256, 300
    a = S.normal((M, Kd), 1.0, S.key(0, "err-gemm-a")).cuda()
    qa, sa = m.fp8_quant_1x128(a)
    b = S.normal((G * Nd, Kd), 0.05, S.key(0, "err-gemm-b")).cuda()
    qb, sb = m.fp8_quant_128x128(b)
    offs = torch.tensor([0, 200, 100, 300], dtype=torch.int32).cuda()
    C = torch.full((M, Nd), float("nan"), dtype=torch.bfloat16).cuda()
    m.fp8_grouped_gemm(qa, sa, qb.view(G, Nd, Kd), sb.view(G, Nd // 128, Kd // 128), offs, m.MOE_EPI_BF16, C=C)
    assert m.device_status() == m.MOE_ERR_DEVICE_DATA
    assert torch.isnan(C.float()).all()                 # nothing was computed or written
    _context_still_works()


def test_combine_reports_out_of_range_rows():
    m = _lib()
    T, d, K = 40, 256, 2
    R = T * K + T
    u = S.normal((T, d), 1.0, S.key(0, "err-comb-u")).cuda()
    y = S.normal((R, d), 1.0, S.key(0, "err-comb-y")).cuda()
    g = torch.full((T, K), 0.5, dtype=torch.float32).cuda()
    dest = torch.arange(T * K, dtype=torch.int32).view(T, K).cuda()
    dest[7, 1] = R
    m.moe_combine(u, y[T * K:], y, g, dest)
    assert m.device_status() == m.MOE_ERR_DEVICE_DATA
    _context_still_works()


def _route_valid(idx, N, K):
    """Every token has K distinct expert ids in [0, N), ascending."""
    idx = idx.cpu().numpy()
    assert idx.shape[1] == K
    assert ((idx >= 0) & (idx < N)).all()
    assert (np.diff(idx, axis=1) > 0).all()
    return idx


@pytest.mark.parametrize("n_groups,topk_groups", [(1, 1), (8, 3)])
def test_route_nan_tokens_and_minus_inf_bias_keep_valid_ids(n_groups, topk_groups):
    """A NaN in a token makes all of its affinities NaN, and a -inf bias makes an
    expert's key -inf; neither may produce an expert id outside [0, N) (the
    selection ranks NaN keys last, ties to the lower index). The other tokens are
    routed as usual and the loads match the ids."""
    m = _lib()
    T, d, N, K = 64, 256, 64, 6
    u = S.normal((T, d), 1.0, S.key(0, "nan-u")).clone()
    u[5, 17] = float("nan")
    u[40, :] = float("nan")
    e = S.normal((N, d), 1.0 / 16, S.key(0, "nan-e"), dtype=torch.float32)
    b = S.uniform((N,), -0.01, 0.01, S.key(0, "nan-b")).clone()
    b[[0, 3, 9, 33]] = float("-inf")
    idx, gates, loads, _ = m.moe_route(u.cuda(), e.cuda(), b.cuda(), K, n_groups, topk_groups)
    assert m.device_status() == m.MOE_OK
    ids = _route_valid(idx, N, K)
    np.testing.assert_array_equal(loads.cpu().numpy(), np.bincount(ids.ravel(), minlength=N))
    # a -inf bias keeps an expert out wherever enough finite keys remain
    ok_rows = np.setdiff1d(np.arange(T), [5, 40])
    assert not np.isin(ids[ok_rows], [0, 3, 9, 33]).any()
    # the same tokens with finite values route exactly as before
    u2 = u.clone()
    u2[5, 17] = 0.0
    u2[40, :] = 0.0
    idx2, _, _, _ = m.moe_route(u2.cuda(), e.cuda(), b.cuda(), K, n_groups, topk_groups)
    np.testing.assert_array_equal(ids[ok_rows], idx2.cpu().numpy()[ok_rows])
    _context_still_works()


def test_route_all_minus_inf_bias_still_picks_k_experts():
    m = _lib()
    T, d, N, K = 16, 128, 32, 8
    u = S.normal((T, d), 1.0, S.key(0, "ninf-u"))
    e = S.normal((N, d), 1.0 / 11, S.key(0, "ninf-e"), dtype=torch.float32)
    b = torch.full((N,), float("-inf"))
    idx, _, loads, _ = m.moe_route(u.cuda(), e.cuda(), b.cuda(), K)
    assert m.device_status() == m.MOE_OK
    ids = _route_valid(idx, N, K)
    # every key ties at -inf: the lowest K ids win
    np.testing.assert_array_equal(ids, np.tile(np.arange(K), (T, 1)))
    assert loads.sum().item() == T * K
    _context_still_works()
