"""Comparison rules shared by the parity tests.

bf16 outputs: the CUDA path and the FP64 oracle round at different points,
so a bf16 output y passes when it is a rounding (either direction) of some
value within a normwise tolerance of the exact result r:

    |y - r| <= tau * max_row|r| + ulp_bf16(max(|r|, |y|))

with tau = 2e-3 (the layer's stated bound on FP8 GEMM / layer outputs) unless a
test asks for a tighter tau. The achieved tau (the smallest that would pass)
is returned so tests can also assert a much tighter figure where the
arithmetic allows it.
"""
from __future__ import annotations

import numpy as np
import torch

# Certified routing gap. The tensor-core gate sums d products (exact in fp32)
# in fp32; at d = 7168 the affinities s = sigmoid(z) measured up to 2.3e-6 away
# from the FP64 oracle's. Two keys each off by that much keep their order when
# their FP64 gap is at least 1e-5, so tokens whose K-th and (K+1)-th keys (or
# last kept and first dropped group scores) are closer than this are the only
# ones allowed to route differently, and only to an equally good set.
ROUTE_DELTA = 1e-5


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7)


def check_bf16(y, r: np.ndarray, tau: float = 2e-3, what: str = "") -> float:
    """Asserts the rule above per row; returns the achieved normwise tau."""
    y = bf16_f64(y) if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    r = np.asarray(r, np.float64)
    assert y.shape == r.shape, (y.shape, r.shape)
    y2, r2 = y.reshape(-1, y.shape[-1]), r.reshape(-1, r.shape[-1])
    M = np.maximum(np.abs(r2).max(axis=1, keepdims=True), 1e-30)
    excess = np.abs(y2 - r2) - ulp_bf16(np.maximum(np.abs(r2), np.abs(y2)))
    achieved = float(np.max(np.maximum(excess, 0.0) / M)) if y2.size else 0.0
    bad = excess > tau * M
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside tolerance {tau}; first at "
                             f"[{i},{j}]: got {y2[i, j]!r}, exact {r2[i, j]!r}, row max {M[i, 0]!r}; "
                             f"achieved tau {achieved:.3e}")
    return achieved


def e4m3_values() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def check_fp8_codes(got: np.ndarray, exp: np.ndarray, dist: np.ndarray, vscaled: np.ndarray, rel_margin=1e-4,
                    what: str = ""):
    """E4M3 codes that a correct fp32 computation may round either way.

    Codes must be equal (as values: +0 and -0 are equal) except where the
    oracle's a/scale lies within rel_margin * max(|v|, 1) of a rounding
    boundary, where the neighbouring code is also accepted. Returns the
    number of accepted differences."""
    vals = e4m3_values()
    g, e = vals[got.astype(np.int64)], vals[exp.astype(np.int64)]
    differ = g != e
    near = dist < rel_margin * np.maximum(np.abs(vscaled), 1.0)
    if np.any(differ & ~near):
        i = np.argwhere(differ & ~near)[0]
        raise AssertionError(f"{what}: {int(np.sum(differ & ~near))} codes differ away from a rounding boundary; "
                             f"first at {tuple(i)}: got {g[tuple(i)]}, expected {e[tuple(i)]}, "
                             f"a/scale {vscaled[tuple(i)]}, boundary distance {dist[tuple(i)]}")
    # where they differ, they are neighbours
    gi, ei = got.astype(np.int64)[differ], exp.astype(np.int64)[differ]
    assert np.all(np.abs((gi & 0x7F) - (ei & 0x7F)) <= 1) or not differ.any(), what
    return int(differ.sum())
