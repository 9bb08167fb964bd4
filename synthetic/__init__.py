"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is shared by the CUDA path's harness (tests, bench) and by the
oracle's callers. It holds none of the layer's arithmetic: it only draws
numbers. Every value comes from a counter-based generator written with
integer and exact-or-IEEE-rounded fp32 torch operations, so the same call gives
bit-identical tensors on the CPU and on a GPU:

  * bits(i)   = h(h(lo(i) ^ h(hi(i) ^ key)) + key), with h the 32-bit
                "lowbias32" integer hash (Chris Wellons, hash-prospector) and
                i the element's flat index;
  * uniform   = (bits >> 8) * 2^-24, then an affine map in fp32;
  * normal    = linear interpolation in a 65,537-entry table of standard
                normal quantiles Q[j] = Phi^-1((j + 1/2) / 65537) (Python's
                statistics.NormalDist, Wichura's AS241), indexed by the top 16
                bits with the low 16 bits as the fraction, then times the
                standard deviation in fp32.  The draws lie in [-4.33, 4.33]
                standard deviations.

The DeepSeek-V3 pages measure nothing on a dataset for this layer; these
configurations are the shapes and distributions the benchmark states
(N(0, std) with std a standard deviation, U(lo, hi), 0.1% outliers x100,
Zipf-skewed expert popularity).
"""
from __future__ import annotations

import functools
import math
import zlib
from dataclasses import dataclass, field
from statistics import NormalDist

import numpy as np
import torch

M32 = 0xFFFFFFFF
_CHUNK = 1 << 24

_QTABLE: dict = {}


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32 without any int64 overflow."""
    c_lo, c_hi = c & 0xFFFF, c >> 16
    return ((x * c_lo) + (((x * c_hi) & 0xFFFF) << 16)) & M32


def _h32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def key(seed: int, *names) -> int:
    """Stable 32-bit stream key for (seed, names...)."""
    text = f"{seed}/" + "/".join(str(n) for n in names)
    return zlib.crc32(text.encode()) & M32


def bits(key_: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """n uniform 32-bit integers (as int64) for flat indices start..start+n-1."""
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    lo = i & M32
    hi = i >> 32
    k = torch.full_like(hi, key_)
    x = _h32(lo ^ _h32(hi ^ k))
    return _h32((x + key_) & M32)


def _qtable(device) -> torch.Tensor:
    dev = torch.device(device)
    t = _QTABLE.get(dev)
    if t is None:
        nd = NormalDist()
        q = [nd.inv_cdf((j + 0.5) / 65537.0) for j in range(65537)]
        t = torch.tensor(q, dtype=torch.float64).to(torch.float32).to(dev)
        _QTABLE[dev] = t
    return t


def _normal_flat(key_: int, start: int, n: int, std: float, device) -> torch.Tensor:
    q = _qtable(device)
    out = torch.empty(n, dtype=torch.float32, device=device)
    s = torch.tensor(std, dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        x = bits(key_, start + c0, c1 - c0, device)
        idx = x >> 16
        frac = (x & 0xFFFF).to(torch.float32) * (1.0 / 65536.0)
        q0 = q[idx]
        q1 = q[idx + 1]
        z = q0 + frac * (q1 - q0)
        out[c0:c1] = z * s
    return out


def normal(shape, std: float, key_: int, device="cpu", dtype=torch.bfloat16, start: int = 0) -> torch.Tensor:
    """Tensor of N(0, std) draws (std is the standard deviation)."""
    n = int(np.prod(shape)) if len(shape) else 1
    z = _normal_flat(key_, start, n, std, device)
    return z.to(dtype).reshape(shape)


def uniform(shape, lo: float, hi: float, key_: int, device="cpu", start: int = 0) -> torch.Tensor:
    """fp32 tensor of U(lo, hi) draws."""
    n = int(np.prod(shape)) if len(shape) else 1
    x = bits(key_, start, n, device)
    f = (x >> 8).to(torch.float32) * (1.0 / 16777216.0)
    lo_t = torch.tensor(lo, dtype=torch.float32, device=device)
    w_t = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    return (lo_t + w_t * f).reshape(shape)


def permutation(n: int, key_: int) -> torch.Tensor:
    """A seeded permutation of 0..n-1 (argsort of unique 64-bit hash keys)."""
    h = bits(key_, 0, n, "cpu")
    k = h * (1 << 20) + torch.arange(n, dtype=torch.int64)
    return torch.argsort(k)


def choose_positions(total: int, count: int, key_: int) -> torch.Tensor:
    """count distinct positions in [0, total), uniform without replacement."""
    h = bits(key_, 0, total, "cpu")
    k = h * (1 << 31) + torch.arange(total, dtype=torch.int64)
    return torch.topk(k, count, largest=False, sorted=True).indices


# --------------------------------------------------------------------------
# Zipf-skewed expert popularity for the full-size layer
# --------------------------------------------------------------------------

def zipf_targets(n_experts: int, k: int, s: float = 1.1, cap: float = 0.5):
    """Per-rank selection probabilities p_r = min(cap, c * r^-s), sum p = k."""
    r = np.arange(1, n_experts + 1, dtype=np.float64)
    lo, hi = 0.0, 100.0
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(cap, c * r ** (-s)).sum() < k:
            lo = c
        else:
            hi = c
    c = 0.5 * (lo + hi)
    return np.minimum(cap, c * r ** (-s)), c


@functools.lru_cache(maxsize=4)
def zipf_norms(n_experts: int, k: int, seed: int = 2, samples: int = 8192, rounds: int = 100):
    """Centroid norms r_i whose expert is picked with Zipf(1.1)-like probability.

    Input shaping only: with u ~ N(0, I) and nearly orthogonal random
    directions, the dot products u.e_i behave as independent N(0, r_i^2)
    scalars, so the norms are fitted on scalar draws. Each round counts how
    often each expert is among the k largest of r_i * g_i over `samples`
    draws, multiplies r_i by (target / observed)^0.2, divides by the median
    and clips to [1/16, 16]. The three hottest targets (capped at 0.5) end
    near 0.44, the most a finite norm can give. Rank 1 goes to expert perm[0],
    and so on, by a seeded permutation. The result is rounded to a 2^-12 grid
    so that it does not depend on the last bit of any host reduction.
    """
    p, _ = zipf_targets(n_experts, k)
    g = normal((samples, n_experts), 1.0, key(seed, "zipf-calibration"), dtype=torch.float32).double().numpy()
    r = np.ones(n_experts)
    for _ in range(rounds):
        z = g * r[None, :]
        top = np.argpartition(-z, k - 1, axis=1)[:, :k]
        f = np.bincount(top.ravel(), minlength=n_experts) / samples
        f = np.maximum(f, 0.5 / samples)
        r = r * (p / f) ** 0.2
        r = np.clip(r / np.median(r), 1.0 / 16.0, 16.0)
    r = np.round(r * 4096.0) / 4096.0
    perm = permutation(n_experts, key(seed, "zipf-rank")).numpy()
    norms = np.empty(n_experts)
    norms[perm] = r
    return norms


# --------------------------------------------------------------------------
# The benchmark's configurations
# --------------------------------------------------------------------------

@dataclass
class LayerShape:
    T: int
    d: int
    N: int          # routed experts
    K: int          # experts per token
    I: int          # SwiGLU intermediate size
    n_groups: int = 1
    topk_groups: int = 1
    gamma: float = 1e-3
    fp8: bool = True
    centroid_f32: bool = True
    name: str = ""
    extra: dict = field(default_factory=dict)


TINY = LayerShape(T=128, d=256, N=16, K=4, I=128, fp8=False, centroid_f32=False, name="tiny-bf16")
ROUTE_V3 = LayerShape(T=16384, d=7168, N=256, K=8, I=2048, name="route-dispatch-v3")
GEMM_V3 = dict(M=4096, K=7168, N=4096, outlier_frac=0.001, outlier_mul=100.0, b_std=0.02)
LAYER_V3 = LayerShape(T=8192, d=7168, N=256, K=8, I=2048, name="layer-v3-fp8")
DECODE_V3 = [LayerShape(T=t, d=7168, N=256, K=8, I=2048, n_groups=8, topk_groups=4,
                        name=f"decode-v3-T{t}") for t in (64, 256)]


def tokens(shape: LayerShape, seed: int = 0, device="cpu", start_token: int = 0, count=None) -> torch.Tensor:
    """u ~ N(0,1) bf16 [count, d] for tokens start_token.. (default: all T)."""
    count = shape.T if count is None else count
    return normal((count, shape.d), 1.0, key(seed, "u", shape.d), device,
                  start=start_token * shape.d)


def grad_out(shape: LayerShape, seed: int = 0, device="cpu", std: float = 1.0) -> torch.Tensor:
    """An incoming gradient dL/dh' ~ N(0, std^2) bf16 [T, d] for the backward pass."""
    return normal((shape.T, shape.d), std, key(seed, "grad-out", shape.d), device)


def bias(shape: LayerShape, seed: int = 0, zero: bool = False, device="cpu") -> torch.Tensor:
    if zero:
        return torch.zeros(shape.N, dtype=torch.float32, device=device)
    return uniform((shape.N,), -0.01, 0.01, key(seed, "bias", shape.N), device)


def centroids(shape: LayerShape, seed: int = 1, zipf: bool = False, device="cpu") -> torch.Tensor:
    """Expert centroids [N, d]: N(0, 1/sqrt(d)), fp32 or bf16; optionally Zipf-scaled."""
    std = 1.0 / math.sqrt(shape.d)
    if not shape.centroid_f32:
        return normal((shape.N, shape.d), std, key(seed, "centroid", shape.N, shape.d), device)
    e = normal((shape.N, shape.d), std, key(seed, "centroid", shape.N, shape.d), device,
               dtype=torch.float32)
    if zipf:
        r = torch.tensor(zipf_norms(shape.N, shape.K), dtype=torch.float32, device=device)
        e = e * r[:, None]
    return e


def expert_weights(shape: LayerShape, e: int, seed: int = 1, device="cpu", dtype=torch.bfloat16):
    """(W1 [I,d], W3 [I,d], W2 [d,I]) of expert e; e == N is the shared expert.

    Standard deviations 1/sqrt(d) for W1, W3 and 1/sqrt(I) for W2 at the V3
    shape; the tiny configuration draws every weight with 1/sqrt(d).
    """
    s13 = 1.0 / math.sqrt(shape.d)
    s2 = 1.0 / math.sqrt(shape.d if not shape.fp8 else shape.I)
    w1 = normal((shape.I, shape.d), s13, key(seed, "w1", e, shape.I, shape.d), device, dtype)
    w3 = normal((shape.I, shape.d), s13, key(seed, "w3", e, shape.I, shape.d), device, dtype)
    w2 = normal((shape.d, shape.I), s2, key(seed, "w2", e, shape.I, shape.d), device, dtype)
    return w1, w3, w2


def gemm_operands(M=4096, K=7168, N=4096, seed: int = 0, device="cpu", outlier_frac=0.001,
                  outlier_mul=100.0, b_std=0.02):
    """Dense FP8-GEMM inputs: A [M,K] N(0,1) bf16 with floor(frac*M*K) entries x100;
    B stored [N,K] (the logical K x N weight, transposed so K is contiguous)."""
    a = normal((M, K), 1.0, key(seed, "gemm-a", M, K), device, torch.float32)
    n_out = int(math.floor(outlier_frac * M * K))
    if n_out:
        pos = choose_positions(M * K, n_out, key(seed, "gemm-outliers", M, K)).to(device)
        flat = a.view(-1)
        flat[pos] = flat[pos] * torch.tensor(outlier_mul, dtype=torch.float32, device=device)
    b = normal((N, K), b_std, key(seed + 1, "gemm-b", N, K), device)
    return a.to(torch.bfloat16), b
