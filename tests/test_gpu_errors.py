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
