"""The quantisers' shortcut for x / scale, checked on the CPU against the IEEE
division it stands in for.

Several kernels compute the E4M3 code of fl32(x / s) as the code of
q0 = fl32(x * fl32(1 / s)), and take the division only where q0 may lie on
the other side of a midpoint between two E4M3 values than fl32(x / s) does:
for |q0| >= 2^-6 when the low 20 fp32 fraction bits read within 8 of 0x80000
(a midpoint of E4M3's normals), for 2^-11 <= |q0| < 2^-6 (E4M3's subnormal
steps and the midpoint 2^-10 between 0 and the smallest subnormal), and for a
scale below the smallest normal float (its reciprocal would not be within
half a unit).

The rule is restated here in numpy float32 (IEEE products, quotients and
reciprocals) and must give the codes of the true quotients (the oracle's
encoder) for every bf16 value under many scales, for random fp32 values, and
for values placed within a few units of every midpoint.
"""
import numpy as np
import torch

import oracle

F32 = np.float32


def shortcut(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    x = np.asarray(x, F32)
    s = np.broadcast_to(np.asarray(s, F32), x.shape)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore", under="ignore"):
        r = np.where(s >= F32(2.0**-126), F32(1.0) / s, F32(0.0)).astype(F32)
        q0 = (x * r).astype(F32)
        bits = (q0.view(np.uint32) & np.uint32(0x7FFFFFFF)).astype(np.int64)
        E = bits >> 23
        near = np.abs((bits & 0xFFFFF) - 0x80000) <= 8
        slow = (r == 0) | ((E >= 116) & (E < 121)) | ((E >= 121) & near)
        return np.where(slow, (x / s).astype(F32), q0)


def exact(x, s):
    with np.errstate(over="ignore", divide="ignore", invalid="ignore", under="ignore"):
        return (np.asarray(x, F32) / np.asarray(s, F32)).astype(F32)


def scale_of(amax):
    return F32(1.0) if amax == 0 else F32(F32(amax) / F32(448.0))


def check(x, s):
    a, b = oracle.e4m3_encode(shortcut(x, s)), oracle.e4m3_encode(exact(x, s))
    bad = np.nonzero(a != b)[0]
    assert bad.size == 0, (f"{bad.size} codes differ, first x={np.asarray(x).ravel()[bad[0]]!r} "
                           f"s={np.broadcast_to(s, np.shape(x)).ravel()[bad[0]]!r}")


def bf16_grid(limit):
    """Every bf16 value of magnitude <= limit, both signs (as fp32)."""
    v = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(F32)
    v = v[v <= limit]
    return np.concatenate([v, -v])


def test_every_bf16_value_under_many_scales():
    rng = np.random.Generator(np.random.PCG64(3))
    amaxes = [448.0, 1.0, 3.140625, 0.0078125, 1e-30, 6e-36, 5e-36, 1e-38, 3e20, 1.7e38]
    mant = rng.integers(0x80, 0x100, 40)
    expo = rng.integers(-60, 60, 40)
    amaxes += [float(m) * 2.0 ** float(e - 7) for m, e in zip(mant, expo)]
    for amax in amaxes:
        a = float(np.asarray(amax, F32).astype(np.float32))
        a = float(((np.asarray([a], F32).view(np.uint32) >> 16) << 16).view(F32)[0])   # a bf16 value
        check(bf16_grid(a), scale_of(a))


def test_random_fp32_values():
    """Products such as the SwiGLU operand are arbitrary fp32 values."""
    rng = np.random.Generator(np.random.PCG64(4))
    for _ in range(20):
        amax = F32(np.exp(rng.uniform(-60, 60)))
        x = (rng.uniform(-1.0, 1.0, 200_000) * np.exp(rng.uniform(-25, 0, 200_000)) * amax).astype(F32)
        x[0] = amax
        check(x, scale_of(amax))


def test_values_next_to_every_midpoint():
    """x placed so that x / s falls within a few units of each midpoint between
    two E4M3 values (and of the ties themselves)."""
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = np.sort(torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy())
    mids = (vals[:-1] + vals[1:]) / 2.0
    mids = np.concatenate([mids, [464.0]])
    rng = np.random.Generator(np.random.PCG64(5))
    scales = [F32(1.0), F32(0.0078125)] + [scale_of(F32(v)) for v in np.exp(rng.uniform(-40, 40, 30))]
    for s in scales:
        base = (mids * np.float64(s)).astype(F32)
        steps = np.arange(-24, 25, dtype=np.int32)
        x = (base.view(np.int32)[:, None] + steps[None, :]).astype(np.int32).view(F32).ravel()
        x = x[np.isfinite(x)]
        check(np.concatenate([x, -x]), s)


def test_values_next_to_the_smallest_midpoints_under_many_scales():
    """Around 2^-10 (between 0 and the smallest subnormal) and the subnormal
    midpoints, under 4000 scales: the rounding of the reciprocal differs from
    scale to scale, so some products land on the other side."""
    rng = np.random.Generator(np.random.PCG64(6))
    s = np.array([scale_of(F32(v)) for v in np.exp(rng.uniform(-60, 60, 4000))], F32)
    mids = np.array([2.0**-10, 1.5 * 2.0**-9, 2.5 * 2.0**-9, 7.5 * 2.0**-9, 1.0625 * 2.0**-6])
    base = (mids[None, :] * s[:, None].astype(np.float64)).astype(F32)
    steps = np.arange(-12, 13, dtype=np.int32)
    x = (base.view(np.int32)[:, :, None] + steps[None, None, :]).view(F32)
    sx = np.broadcast_to(s[:, None, None], x.shape)
    check(x.ravel(), sx.ravel())
