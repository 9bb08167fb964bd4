"""Pins for the oracle's number formats: E4M3 and bf16 rounding.

The oracle's encoder searches a table it builds from the OCP E4M3 definition;
these tests hold it against torch's float8_e4m3fn conversion (a library
routine), against exhaustive nearest-code search, and against closed forms.
"""
import numpy as np
import pytest
import torch

import oracle


def _torch_e4m3_codes(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_values()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    # closed forms of the format: max 448, min normal 2^-6, min subnormal 2^-9
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])


def test_codes_reencode_to_themselves():
    vals = oracle.e4m3_values()
    codes = np.arange(256)
    finite = ~np.isnan(vals)
    enc = oracle.e4m3_encode(vals[finite].astype(np.float32))
    np.testing.assert_array_equal(enc, codes[finite].astype(np.uint8))


@pytest.mark.parametrize("exp", [-12, -10, -9, -7, -6, -5, 0, 3, 7, 8])
def test_encoder_matches_torch_whole_binade(exp):
    # every fp32 value of the binade [2^exp, 2^(exp+1)), both signs
    m = np.arange(1 << 23, dtype=np.uint32)
    bits = ((np.uint32(exp + 127) << 23) | m).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.abs(v) <= 448.0]
    for s in (1.0, -1.0):
        x = (v * np.float32(s)).astype(np.float32)
        np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_e4m3_codes(x))


def test_encoder_matches_torch_random_and_ties():
    rng = np.random.Generator(np.random.PCG64(7))
    x = (rng.standard_normal(2_000_000) * rng.choice([1e-3, 0.1, 1.0, 30.0, 200.0], 2_000_000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_e4m3_codes(x))
    # exact midpoints between adjacent codes round to the even code
    vals = oracle.e4m3_values()[:127]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)
    enc = oracle.e4m3_encode(mids).astype(int)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    np.testing.assert_array_equal(enc, expect)
    np.testing.assert_array_equal(enc, _torch_e4m3_codes(mids))


def test_encoder_is_nearest_code_brute_force():
    vals = oracle.e4m3_values()
    codes = np.arange(256)
    finite = ~np.isnan(vals)
    rng = np.random.Generator(np.random.PCG64(3))
    x = rng.uniform(-448, 448, 3000).astype(np.float32)
    x[:200] = (rng.integers(-3000, 3000, 200) * 2.0 ** -12).astype(np.float32)  # subnormal range
    enc = oracle.e4m3_encode(x)
    for xi, c in zip(x, enc):
        same_sign = finite & ((codes >= 128) == bool(np.signbit(xi)))
        d = np.abs(vals - float(xi))
        d[~same_sign] = np.inf
        best = codes[d == d.min()]
        if len(best) == 1:
            assert c == best[0]
        else:
            assert len(best) == 2 and c == best[best % 2 == 0][0]


def test_saturation_and_signed_zero():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, -1e30, -0.0, 0.0, -1e-20], np.float32)
    enc = oracle.e4m3_encode(x)
    np.testing.assert_array_equal(enc, np.array([0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x80], np.uint8))


def test_bf16_round_matches_torch_on_fp32_inputs():
    rng = np.random.Generator(np.random.PCG64(11))
    x = (rng.standard_normal(1_000_000) * 10.0 ** rng.integers(-6, 6, 1_000_000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_is_single_rounding():
    # 1 + 2^-8 + 2^-30: nearest bf16 is 1 + 2^-7; rounding to fp32 first would
    # give the tie 1 + 2^-8, which then goes to even (1.0).
    x = np.array([1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -30)])
    got = oracle.bf16_value(oracle.bf16_round(x))
    np.testing.assert_array_equal(got, [1 + 2 ** -7, 1.0, 1 + 2 * 2 ** -7, -(1 + 2 ** -7)])


def test_boundary_distance():
    L = oracle.lib()
    # codes around 1.0 are 0.9375, 1.0, 1.125: boundaries at 0.96875 and 1.0625
    assert L.oracle_e4m3_boundary_distance(1.0) == 0.03125
    assert L.oracle_e4m3_boundary_distance(1.0625) == 0.0   # exactly a midpoint
    assert L.oracle_e4m3_boundary_distance(440.0) == 8.0    # 432 is the boundary between 416 and 448
