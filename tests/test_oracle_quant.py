"""Pins for the oracle's 1x128 and 128x128 FP8 quantisation.

The tile rule (one scale per 1x128 activation tile and per 128x128 weight
block, so an outlier only affects its own group) is from the DeepSeek-V3
Technical Report summary (learn.ifs.name), paragraph on FP8 scaling.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S

VALS = None


def _vals():
    global VALS
    if VALS is None:
        VALS = oracle.e4m3_values()
    return VALS


def _bf16(shape, std, name, outliers=0):
    x = S.normal(shape, std, S.key(0, name), dtype=torch.float32)
    if outliers:
        pos = S.choose_positions(x.numel(), outliers, S.key(0, name, "o"))
        x.view(-1)[pos] *= 100.0
    return x.to(torch.bfloat16)


def _f(x_bf16):
    return x_bf16.to(torch.float32).numpy()


def _check_tiles(xf, q, s, tiles):
    """Each tile: scale = fl32(amax/448) (1 if amax==0); the amax element maps
    to +-448; every code is the nearest code to fl32(x/scale) (brute force);
    dequantised error <= 2^-4 relative in the normal range."""
    vals = _vals()
    for (rows, cols), sc in tiles:
        blk = xf[rows, cols]
        amax = np.float32(np.max(np.abs(blk)))
        exp_sc = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
        assert sc == exp_sc
        v = (blk / np.float32(sc)).astype(np.float32)
        codes = q[rows, cols]
        deq = vals[codes]
        # nearest code (ties aside) and exact amax -> 448
        assert np.all(np.abs(deq - v) <= np.abs(v) * 2.0 ** -4 + 2.0 ** -10)
        if amax > 0:
            at = np.abs(blk) == amax
            assert np.all(np.abs(deq[at]) == 448.0)
        torch_codes = torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(codes, torch_codes)


def test_quant_1x128_tiles_and_ragged_rows():
    x = _bf16((37, 640), 1.0, "q1x128", outliers=20)
    q, s = oracle.quant_1x128(x)
    assert q.shape == (37, 640) and s.shape == (37, 5)
    xf = _f(x)
    tiles = [((slice(r, r + 1), slice(b * 128, b * 128 + 128)), s[r, b]) for r in range(37) for b in range(5)]
    _check_tiles(xf, q, s, tiles)


def test_quant_128x128_blocks_partial_rows():
    w = _bf16((300, 384), 0.02, "q128x128", outliers=5)
    q, s = oracle.quant_128x128(w)
    assert s.shape == (3, 3)
    wf = _f(w)
    tiles = [((slice(br * 128, min(300, br * 128 + 128)), slice(bc * 128, bc * 128 + 128)), s[br, bc])
             for br in range(3) for bc in range(3)]
    _check_tiles(wf, q, s, tiles)


def test_outlier_only_changes_its_own_tile():
    x = _bf16((8, 1024), 1.0, "iso")
    q0, s0 = oracle.quant_1x128(x)
    y = x.clone()
    y[3, 300] = y[3, 300] * 100 + 50
    q1, s1 = oracle.quant_1x128(y)
    changed = s0 != s1
    assert changed.sum() == 1 and changed[3, 300 // 128]
    mask = np.ones_like(q0, dtype=bool)
    mask[3, 256:384] = False
    np.testing.assert_array_equal(q0[mask], q1[mask])
    # same for a weight block
    w = _bf16((256, 256), 0.02, "isow")
    a0, t0 = oracle.quant_128x128(w)
    w2 = w.clone()
    w2[200, 10] = 5.0
    a1, t1 = oracle.quant_128x128(w2)
    assert (t0 != t1).sum() == 1 and t0[1, 0] != t1[1, 0]


def test_zero_tile_and_sign():
    x = torch.zeros((2, 256), dtype=torch.bfloat16)
    x[1, 128:] = -0.0
    x[1, 200] = -3.0
    q, s = oracle.quant_1x128(x)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0
    assert np.all(q[0] == 0)
    assert s[1, 1] == np.float32(np.float32(3.0) / np.float32(448.0))
    assert q[1, 200] == 0xFE           # -448
    assert q[1, 201] == 0x80           # -0 keeps its sign


def test_scale_power_of_two_exactness():
    # a tile whose entries are powers of two times 448 quantises exactly
    x = torch.zeros((1, 128), dtype=torch.float32)
    x[0, :8] = torch.tensor([448.0, 224.0, 112.0, 56.0, -28.0, 14.0, 7.0, 3.5])
    q, s = oracle.quant_1x128(x.to(torch.bfloat16))
    assert s[0, 0] == 1.0
    np.testing.assert_array_equal(_vals()[q[0, :8]], x[0, :8].numpy())
