"""FP64 CPU oracle for the DeepSeekMoE layer: forward, backward and training
step (test infrastructure).

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this package. It wraps the plain C file `moe_oracle.c`
(compiled here with gcc, no fast-math, no FP contraction) through ctypes and
composes its pieces into the layer. It shares no code with the CUDA library
and never imports it.

Parity pins: every function here is checked in tests/test_oracle_*.py and
tests/test_golden_pages.py against something other than itself (closed forms,
brute force with numpy, torch's float8_e4m3fn conversion, invariants, the
figures the pages print). The composed layer is checked against an
independent brute force on a tiny layer; the pages print no worked example at
the full V3 shape, so the full-size value rests on those pins. The backward
pass (tests/test_oracle_backward.py) is checked, in its FP64 form, against
finite differences of an independent forward, and in its FP8 form against
the FP64 form on block-scaled inputs; the training step as a descent step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (next to it) if stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            i64, i32, dbl, flt = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
            vp = ctypes.c_void_p
            sig = {
                "oracle_threads": (i32, []),
                "oracle_init": (None, []),
                "oracle_bf16_value": (dbl, [ctypes.c_uint16]),
                "oracle_bf16_round": (ctypes.c_uint16, [dbl]),
                "oracle_e4m3_value": (dbl, [ctypes.c_uint8]),
                "oracle_e4m3_encode": (ctypes.c_uint8, [flt]),
                "oracle_e4m3_boundary_distance": (dbl, [flt]),
                "oracle_bf16_round_array": (None, [vp, i64, vp]),
                "oracle_e4m3_encode_array": (None, [vp, i64, vp]),
                "oracle_quant_1x128": (None, [vp, i64, i64, vp, vp]),
                "oracle_quant_1x128_f32": (None, [vp, i64, i64, vp, vp]),
                "oracle_quant_128x128": (None, [vp, i64, i64, vp, vp]),
                "oracle_route": (None, [vp, i64, i64, vp, vp, vp, i32, i32, i32, i32, dbl,
                                        vp, vp, vp, vp, vp, vp]),
                "oracle_permute": (None, [vp, i64, i32, i32, vp, vp, vp]),
                "oracle_fp8_gemm": (None, [vp, vp, vp, vp, i64, i64, i64, vp]),
                "oracle_bf16_gemm": (None, [vp, vp, i64, i64, i64, vp]),
                "oracle_swiglu": (None, [vp, vp, i64, vp]),
                "oracle_swiglu_quant": (None, [vp, vp, i64, i64, vp, vp, vp, vp]),
                "oracle_combine": (None, [vp, vp, vp, vp, vp, i64, i64, i32, vp]),
                "oracle_bias_update": (None, [vp, vp, i32, i64, i32, flt]),
                "oracle_seq_balance": (None, [vp, vp, i64, i32, i32, i64, vp, vp, vp]),
                "oracle_quant_128x1": (None, [vp, i64, i64, vp, vp]),
                "oracle_fp8_gemm_kscaled": (None, [vp, vp, vp, vp, i64, i64, i64, vp]),
                "oracle_quant_128x128_f32": (None, [vp, i64, i64, vp, vp]),
                "oracle_swiglu_backward": (None, [vp, vp, vp, i64, vp, vp]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            L.oracle_init()
            _lib = L
        return _lib


def threads() -> int:
    return int(lib().oracle_threads())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (or pass uint16 through)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# formats
# --------------------------------------------------------------------------

def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits of x rounded once, to nearest even, from FP64."""
    flat = _c(np.asarray(x, dtype=np.float64).ravel(), np.float64)
    out = np.empty(flat.size, np.uint16)
    lib().oracle_bf16_round_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(x))


def e4m3_values() -> np.ndarray:
    """The 256 code values (NaN for 0x7F / 0xFF)."""
    L = lib()
    return np.array([L.oracle_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """E4M3 codes of fp32 values (nearest, ties to even, saturating)."""
    flat = _c(np.asarray(v, dtype=np.float32).ravel(), np.float32)
    out = np.empty(flat.size, np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(v))


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------

def quant_1x128(x_bf16) -> tuple[np.ndarray, np.ndarray]:
    """(q uint8 [R,C], scales fp32 [R, C/128]) from bf16 [R,C]."""
    x = as_bf16_bits(x_bf16)
    R, C = x.shape
    assert C % 128 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 128), np.float32)
    lib().oracle_quant_1x128(_ptr(x), R, C, _ptr(q), _ptr(s))
    return q, s


def quant_1x128_f32(x: np.ndarray):
    x = _c(x, np.float32)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 128), np.float32)
    lib().oracle_quant_1x128_f32(_ptr(x), R, C, _ptr(q), _ptr(s))
    return q, s


def quant_128x128(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """(q uint8 [R,C], scales fp32 [ceil(R/128), C/128]) from bf16 [R,C]."""
    w = as_bf16_bits(w_bf16)
    R, C = w.shape
    assert C % 128 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty(((R + 127) // 128, C // 128), np.float32)
    lib().oracle_quant_128x128(_ptr(w), R, C, _ptr(q), _ptr(s))
    return q, s


# --------------------------------------------------------------------------
# routing, permutation, bias
# --------------------------------------------------------------------------

class Route:
    def __init__(self, topk_idx, gates, scores, key_gap, loads, near_tie):
        self.topk_idx, self.gates, self.scores = topk_idx, gates, scores
        self.key_gap, self.loads, self.near_tie = key_gap, loads, near_tie


def route(u_bf16, centroids, bias: np.ndarray, K: int, n_groups: int = 1, topk_groups: int = 1,
          delta: float = 0.0, want_scores: bool = False) -> Route:
    """Sigmoid affinities, biased top-K (optionally group-limited), gates, loads.

    centroids: fp32 numpy/torch array, or a bf16 torch tensor / uint16 array.
    """
    u = as_bf16_bits(u_bf16)
    T, d = u.shape
    cf = cb = None
    import torch
    if isinstance(centroids, torch.Tensor) and centroids.dtype == torch.bfloat16:
        cb = as_bf16_bits(centroids)
    elif isinstance(centroids, np.ndarray) and centroids.dtype == np.uint16:
        cb = centroids
    else:
        cf = _c(centroids.cpu().numpy() if isinstance(centroids, torch.Tensor) else centroids, np.float32)
    N = (cf if cf is not None else cb).shape[0]
    b = _c(bias.cpu().numpy() if isinstance(bias, torch.Tensor) else bias, np.float32)
    idx = np.empty((T, K), np.int32)
    g = np.empty((T, K), np.float64)
    s = np.empty((T, N), np.float64) if want_scores else None
    gap = np.empty(T, np.float64)
    loads = np.empty(N, np.int32)
    near = np.empty(T, np.int32)
    lib().oracle_route(_ptr(u), T, d, _ptr(cf), _ptr(cb), _ptr(b), N, K, n_groups, topk_groups,
                       float(delta), _ptr(idx), _ptr(g), _ptr(s), _ptr(gap), _ptr(loads), _ptr(near))
    return Route(idx, g, s, gap, loads, near.astype(bool))


def permute(topk_idx: np.ndarray, N: int):
    """(offsets [N+1], perm_token [T*K], dest_row [T,K]) by stable counting sort."""
    idx = _c(topk_idx, np.int32)
    T, K = idx.shape
    off = np.empty(N + 1, np.int32)
    perm = np.empty(T * K, np.int32)
    dest = np.empty((T, K), np.int32)
    lib().oracle_permute(_ptr(idx), T, N, K, _ptr(off), _ptr(perm), _ptr(dest))
    return off, perm, dest


def bias_update(bias: np.ndarray, loads: np.ndarray, T: int, K: int, gamma: float) -> np.ndarray:
    b = _c(bias, np.float32).copy()
    ld = _c(loads, np.int32)
    lib().oracle_bias_update(_ptr(b), _ptr(ld), b.size, T, K, float(np.float32(gamma)))
    return b


def seq_balance(scores: np.ndarray, topk_idx: np.ndarray, K: int, seq_len: int):
    """Sequence-wise balance statistics (see moe_oracle.c): per sequence of
    seq_len consecutive tokens (the last may be shorter), the loads [S, N], the
    mean normalised affinities P [S, N] and sum_i f_i P_i [S]."""
    sc = _c(scores, np.float64)
    idx = _c(topk_idx, np.int32)
    T, N = sc.shape
    S = (T + seq_len - 1) // seq_len
    loads = np.empty((S, N), np.int32)
    prob = np.empty((S, N), np.float64)
    stat = np.empty(S, np.float64)
    lib().oracle_seq_balance(_ptr(sc), _ptr(idx), T, N, K, seq_len, _ptr(loads), _ptr(prob), _ptr(stat))
    return loads, prob, stat


# --------------------------------------------------------------------------
# GEMMs, activation, combine
# --------------------------------------------------------------------------

def fp8_gemm(qa, sa, qb, sb) -> np.ndarray:
    """FP64 C [M,Nd] of the block-scaled FP8 product (see moe_oracle.c)."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float32), _c(sb, np.float32)
    M, Kd = qa.shape
    Nd = qb.shape[0]
    C = np.empty((M, Nd), np.float64)
    lib().oracle_fp8_gemm(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, Nd, Kd, _ptr(C))
    return C


def bf16_gemm(a_bf16, b_bf16) -> np.ndarray:
    a, b = as_bf16_bits(a_bf16), as_bf16_bits(b_bf16)
    M, Kd = a.shape
    Nd = b.shape[0]
    C = np.empty((M, Nd), np.float64)
    lib().oracle_bf16_gemm(_ptr(a), _ptr(b), M, Nd, Kd, _ptr(C))
    return C


def swiglu(h1: np.ndarray, h3: np.ndarray) -> np.ndarray:
    h1, h3 = _c(h1, np.float64), _c(h3, np.float64)
    a = np.empty_like(h1)
    lib().oracle_swiglu(_ptr(h1), _ptr(h3), h1.size, _ptr(a))
    return a


def swiglu_quant(h1: np.ndarray, h3: np.ndarray):
    """(q [R,I], scales [R,I/128], boundary distance [R,I], a/scale [R,I])."""
    h1, h3 = _c(h1, np.float64), _c(h3, np.float64)
    R, I = h1.shape
    q = np.empty((R, I), np.uint8)
    s = np.empty((R, I // 128), np.float32)
    dist = np.empty((R, I), np.float64)
    v = np.empty((R, I), np.float64)
    lib().oracle_swiglu_quant(_ptr(h1), _ptr(h3), R, I, _ptr(q), _ptr(s), _ptr(dist), _ptr(v))
    return q, s, dist, v


def combine(u_bf16, y_shared_bf16, y_bf16, gates: np.ndarray, dest_row: np.ndarray) -> np.ndarray:
    u = as_bf16_bits(u_bf16)
    ys = None if y_shared_bf16 is None else as_bf16_bits(y_shared_bf16)
    y = as_bf16_bits(y_bf16)
    g = _c(gates, np.float64)
    dr = _c(dest_row, np.int32)
    T, d = u.shape
    K = g.shape[1]
    out = np.empty((T, d), np.float64)
    lib().oracle_combine(_ptr(u), _ptr(ys), _ptr(y), _ptr(g), _ptr(dr), T, d, K, _ptr(out))
    return out


# --------------------------------------------------------------------------
# the layer, composed from the pieces above
# --------------------------------------------------------------------------

def expert_ffn_fp8(xq, xs, w1, w3, w2, want_detail: bool = False):
    """One SwiGLU expert on FP8 rows: y = W2 (silu(W1 x) * W3 x).

    xq/xs: the rows' E4M3 codes [R,d] and 1x128 scales [R,d/128];
    w1, w3 [I,d] and w2 [d,I] bf16 weights, quantised here per 128x128 block.
    The intermediate is re-quantised per 1x128 tile; y is FP64 [R,d].
    """
    q1, s1 = quant_128x128(w1)
    q3, s3 = quant_128x128(w3)
    q2, s2 = quant_128x128(w2)
    h1 = fp8_gemm(xq, xs, q1, s1)
    h3 = fp8_gemm(xq, xs, q3, s3)
    aq, as_, dist, v = swiglu_quant(h1, h3)
    y = fp8_gemm(aq, as_, q2, s2)
    if want_detail:
        return y, dict(aq=aq, as_=as_, dist=dist, v=v, q2=q2, s2=s2)
    return y


def expert_ffn_bf16(x_bf16, w1, w3, w2):
    """One SwiGLU expert in bf16 with exact products: h = x W^T in FP64,
    a = silu(h1) * h3 rounded to bf16 (where the bf16 path stores it),
    y = a W2^T in FP64."""
    h1 = bf16_gemm(x_bf16, w1)
    h3 = bf16_gemm(x_bf16, w3)
    a = bf16_round(swiglu(h1, h3))
    return bf16_gemm(a, w2)


def layer_tokens(u_bf16, centroids, bias, K, expert_weights, tokens, fp8=True, n_groups=1, topk_groups=1,
                 delta=0.0, route_all=None):
    """h' in FP64 for the listed tokens (nlp-lineage page, "The notation"):

        h'_t = u_t + FFN_shared(u_t) + sum_k g_{t,k} FFN_{idx[t,k]}(u_t)

    expert_weights(e) -> (w1, w3, w2) bf16 (e = N is the shared expert).
    Routing is the oracle's own (route_all, a Route of all tokens, may be
    passed in to avoid recomputing it). The FP8 path quantises each token row
    per 1x128 tile, every weight per 128x128 block and the intermediate per
    1x128 tile; the bf16 path rounds the intermediate and y to bf16 where the
    bf16 kernels store them. Returns (h' [n, d], route of all tokens, and per
    token the expert outputs' boundary-distance details for the FP8 path).
    """
    import torch
    tokens = np.asarray(tokens, dtype=np.int64)
    r = route_all if route_all is not None else route(u_bf16, centroids, bias, K, n_groups, topk_groups, delta)
    u_bits = as_bf16_bits(u_bf16)[tokens]
    T_s, d = u_bits.shape
    N = (centroids.shape[0])
    idx = r.topk_idx[tokens]
    g = r.gates[tokens]
    if fp8:
        xq, xs = quant_1x128(u_bits)
    y_tok = np.zeros((T_s, K, d))
    y_sh = None
    detail = {}
    for e in range(N + 1):
        if e == N:
            rows = np.arange(T_s)
            ks = None
        else:
            rows, ks = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        w1, w3, w2 = expert_weights(e)
        if fp8:
            y, det = expert_ffn_fp8(xq[rows], xs[rows], w1, w3, w2, want_detail=True)
            detail[e] = (rows, det)
        else:
            y = bf16_value(bf16_round(expert_ffn_bf16(u_bits[rows], w1, w3, w2)))
        if fp8:
            y = bf16_value(bf16_round(y))       # the CUDA path stores expert outputs as bf16
        if e == N:
            y_sh = y
        else:
            y_tok[rows, ks] = y
    h = bf16_value(u_bits) + y_sh + np.einsum("tk,tkd->td", g, y_tok)
    return h, r, detail


# --------------------------------------------------------------------------
# backward pass and training step (readings in moe_oracle.c, [train])
# --------------------------------------------------------------------------

def quant_128x1(x: np.ndarray):
    """(q uint8 [C, Rp], scales fp32 [Rp/128, C]) from fp32 x [R, C]: one scale
    per (128 consecutive rows, column); Rp = R rounded up to 128, the missing
    rows counting as zeros; q holds the columns of x as its rows."""
    x = _c(x, np.float32)
    R, C = x.shape
    Rp = (R + 127) // 128 * 128
    q = np.empty((C, Rp), np.uint8)
    s = np.empty((Rp // 128, C), np.float32)
    lib().oracle_quant_128x1(_ptr(x), R, C, _ptr(q), _ptr(s))
    return q, s


def fp8_gemm_kscaled(qa, sa, qb, sb) -> np.ndarray:
    """FP64 C [M, Nd] = the weight-gradient product of qa [M, Kp] and qb [Nd, Kp]
    with scales sa [Kp/128, M], sb [Kp/128, Nd] (see moe_oracle.c)."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float32), _c(sb, np.float32)
    M, Kp = qa.shape
    Nd = qb.shape[0]
    C = np.empty((M, Nd), np.float64)
    lib().oracle_fp8_gemm_kscaled(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, Nd, Kp, _ptr(C))
    return C


def quant_128x128_f32(w: np.ndarray):
    """(q uint8 [R,C], scales fp32 [ceil(R/128), C/128]) from fp32 w [R,C]."""
    w = _c(w, np.float32)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty(((R + 127) // 128, C // 128), np.float32)
    lib().oracle_quant_128x128_f32(_ptr(w), R, C, _ptr(q), _ptr(s))
    return q, s


def swiglu_backward(h1: np.ndarray, h3: np.ndarray, da: np.ndarray):
    """(dh1, dh3) in FP64 for a = silu(h1) * h3."""
    h1, h3, da = _c(h1, np.float64), _c(h3, np.float64), _c(da, np.float64)
    dh1, dh3 = np.empty_like(h1), np.empty_like(h1)
    lib().oracle_swiglu_backward(_ptr(h1), _ptr(h3), _ptr(da), h1.size, _ptr(dh1), _ptr(dh3))
    return dh1, dh3


def _f32(w) -> np.ndarray:
    """fp32 numpy values of a weight given as a torch tensor (bf16 / fp32) or array."""
    import torch
    if isinstance(w, torch.Tensor):
        return w.detach().float().cpu().numpy()
    return np.asarray(w, np.float32)


def _r32(x: np.ndarray) -> np.ndarray:
    """FP64 -> fp32, one rounding to nearest."""
    return np.asarray(x, np.float64).astype(np.float32)


def _bf(x: np.ndarray) -> np.ndarray:
    """FP64 values of x rounded once to bf16."""
    return bf16_value(bf16_round(x))


class Backward:
    """Everything layer_backward computes (FP64 unless stated):
    h [T,d] (the forward output, before its bf16 rounding), du [T,d],
    dw1, dw3 [N+1, I, d], dw2 [N+1, d, I], de [N, d], dg, dz [T,K],
    route (the oracle's routing), rows[e] (token ids of expert e's rows in
    permuted order) and per-expert intermediates in `inter[e]`."""


def layer_backward(u_bf16, centroids, bias, K, expert_weights, G_bf16, n_groups=1, topk_groups=1, fp8=True,
                   route_all=None, stack=True, wgrad_experts=None) -> Backward:
    """Gradient of L = sum(G * h') for the layer h' (nlp-lineage page, "The
    notation") with the expert choice held fixed (readings in moe_oracle.c,
    [train]):

      combine      dY_r = g_{t,k} G_t (routed row r of (t,k)), dY = G_t (shared),
                   dg_{t,k} = G_t . y_{row(t,k)}
      expert e     dA = dY W2,  (dH1, dH3) = SwiGLU'(H1, H3) dA,  dX = dH1 W1 + dH3 W3
                   dW2 = dY^T A,  dW1 = dH1^T X,  dW3 = dH3^T X   (X = u of the rows)
      gates        with S = sum_k s_k and c = sum_k g_k dg_k:
                   dz_{t,k} = (dg_{t,k} - c) / S * s'(z_k), s'(z) = s (1 - s)
                   = e^-|z| / (1 + e^-|z|)^2 from the logit z = u . e
      tokens       du_t = G_t + dX_shared,t + sum_k dX_{row(t,k)} + sum_k dz_{t,k} e_{idx}
      centroids    de_i = sum over (t,k) routed to i of dz_{t,k} u_t

    fp8=True follows the FP8 path's storage and quantisation points: the
    forward keeps H = X W13^T (FP8 product) rounded to bf16 and its expert
    outputs y in bf16; dY = g G_t is quantised per 1x128 tile for dA = dY W2
    (W2's forward 128x128 blocks, transposed) -- the tile rule is
    scale-invariant, so that is G_t's codes with g times G_t's scales
    (fl32(g s)) -- and dA is stored in bf16; for the weight gradient dY is
    formed in fp32 (fl32(g G));
    dH is computed from the stored H and dA and stored in bf16, quantised per
    1x128 tile for dX = dH W13 (bf16 out); the weight gradients quantise both
    operands per (128 rows of the expert, column) -- dY, A recomputed in fp32
    from the stored H, dH, and u -- and come out in fp32; du is rounded to
    bf16 once at the end (the value returned is before that rounding).
    fp8=False is the same chain with no quantisation and no rounding at all
    (FP64 throughout), the form the finite-difference pins check.

    expert_weights(e) -> (w1 [I,d], w3 [I,d], w2 [d,I]) as bf16 torch tensors or
    fp32 arrays; e = N is the shared expert; it is called only for experts
    with rows. stack=False returns dw1, dw3, dw2 as dicts over the experts
    with rows (for samples of a large layer) instead of stacked arrays;
    wgrad_experts (a set of expert ids, None = all) limits the weight
    gradients to those experts (the others come out as zeros / absent).
    """
    import torch
    u_bits = as_bf16_bits(u_bf16)
    uv = bf16_value(u_bits)
    Gv = bf16_value(as_bf16_bits(G_bf16))
    T, d = uv.shape
    if isinstance(centroids, torch.Tensor) and centroids.dtype == torch.bfloat16:
        Ev = bf16_value(as_bf16_bits(centroids))
    else:
        Ev = _f32(centroids).astype(np.float64)
    N = Ev.shape[0]
    r = route_all if route_all is not None else route(u_bf16, centroids, bias, K, n_groups, topk_groups,
                                                      want_scores=True)
    idx, g, s = r.topk_idx, r.gates, r.scores
    off, perm, dest = permute(idx, N)
    # gate of each routed row
    rgate = np.empty(T * K)
    rgate[dest.ravel()] = g.ravel()
    out = Backward()
    out.route, out.offsets, out.perm_token, out.dest_row = r, off, perm, dest
    out.rows, out.inter = {}, {}
    I = None
    Y_rows = np.zeros((T * K, d))
    Y_sh = None
    dX_rows = np.zeros((T * K, d))
    dX_sh = None
    dW1, dW3, dW2 = {}, {}, {}
    I = _f32(expert_weights(N)[0]).shape[0]
    for e in range(N + 1):
        if e == N:
            rows = np.arange(T)
            toks = rows
            gr = np.ones(T)
        else:
            rows = np.arange(off[e], off[e + 1])
            toks = perm[rows]
            gr = rgate[rows]
        out.rows[e] = toks
        n = toks.size
        if n == 0:   # an expert without rows: no product, zero weight gradients
            continue
        w1, w3, w2 = (_f32(w) for w in expert_weights(e))
        X = uv[toks]
        if fp8:
            xq, xs = quant_1x128(u_bits[toks])
            (q1, s1), (q3, s3), (q2, s2) = (quant_128x128_f32(w) for w in (w1, w3, w2))
            H1, H3 = fp8_gemm(xq, xs, q1, s1), fp8_gemm(xq, xs, q3, s3)
            aq, as_, _, _ = swiglu_quant(H1, H3)
            Y = _bf(fp8_gemm(aq, as_, q2, s2))
            Ht1, Ht3 = _bf(H1), _bf(H3)
            dY = _r32(gr[:, None] * Gv[toks])
            # the 1x128 rule on g G_t: scale-invariant, so G_t's codes and g times its scales
            qy, sg = quant_1x128(as_bf16_bits(G_bf16)[toks])
            sy = _r32(gr[:, None] * sg.astype(np.float64))
            dA = _bf(fp8_gemm(qy, sy, q2.T, s2.T))
            dH1, dH3 = swiglu_backward(Ht1, Ht3, dA)
            dHt1, dHt3 = _bf(dH1), _bf(dH3)
            qh1, sh1 = quant_1x128(bf16_round(dHt1))
            qh3, sh3 = quant_1x128(bf16_round(dHt3))
            dX = _bf(fp8_gemm(qh1, sh1, q1.T, s1.T) + fp8_gemm(qh3, sh3, q3.T, s3.T))
            out.inter[e] = dict(Ht1=Ht1, Ht3=Ht3, Y=Y, dY=dY, dA=dA, dHt1=dHt1, dHt3=dHt3, dX=dX)
            if wgrad_experts is not None and e not in wgrad_experts:
                if e == N:
                    Y_sh, dX_sh = Y, dX
                else:
                    Y_rows[rows] = Y
                    dX_rows[rows] = dX
                continue
            # weight gradients: operands quantised per (128 rows, column)
            A32 = _r32(swiglu(Ht1, Ht3))
            yq_t, ys_t = quant_128x1(dY)
            aq_t, as_t = quant_128x1(A32)
            xq_t, xs_t = quant_128x1(X.astype(np.float32))
            hq1_t, hs1_t = quant_128x1(dHt1.astype(np.float32))
            hq3_t, hs3_t = quant_128x1(dHt3.astype(np.float32))
            dW2[e] = fp8_gemm_kscaled(yq_t, ys_t, aq_t, as_t)
            dW1[e] = fp8_gemm_kscaled(hq1_t, hs1_t, xq_t, xs_t)
            dW3[e] = fp8_gemm_kscaled(hq3_t, hs3_t, xq_t, xs_t)
        else:
            W1, W3, W2 = (w.astype(np.float64) for w in (w1, w3, w2))
            H1, H3 = X @ W1.T, X @ W3.T
            A = swiglu(H1, H3)
            Y = A @ W2.T
            dY = gr[:, None] * Gv[toks]
            dA = dY @ W2
            dH1, dH3 = swiglu_backward(H1, H3, dA)
            dX = dH1 @ W1 + dH3 @ W3
            if wgrad_experts is None or e in wgrad_experts:
                dW2[e] = dY.T @ A
                dW1[e] = dH1.T @ X
                dW3[e] = dH3.T @ X
            out.inter[e] = dict(Ht1=H1, Ht3=H3, Y=Y, dY=dY, dA=dA, dHt1=dH1, dHt3=dH3, dX=dX)
        if e == N:
            Y_sh, dX_sh = Y, dX
        else:
            Y_rows[rows] = Y
            dX_rows[rows] = dX
    rows_tk = dest                                   # [T, K] row of each (t, k)
    Yk = Y_rows[rows_tk]                             # [T, K, d]
    out.h = uv + Y_sh + np.einsum("tk,tkd->td", g, Yk)
    dg = np.einsum("td,tkd->tk", Gv, Yk)
    s_sel = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    S = s_sel.sum(axis=1, keepdims=True)
    c = (g * dg).sum(axis=1, keepdims=True)
    # the sigmoid's derivative s (1 - s), from the logit z = u . e (no cancellation near s = 1)
    z = np.einsum("td,tkd->tk", uv, Ev[idx])
    ez = np.exp(-np.abs(z))
    dz = (dg - c) / S * (ez / (1.0 + ez) ** 2)
    du = Gv + dX_sh + dX_rows[rows_tk].sum(axis=1) + np.einsum("tk,tkd->td", dz, Ev[idx])
    de = np.zeros((N, d))
    for i in range(N):
        tt, kk = np.nonzero(idx == i)
        if tt.size:
            de[i] = (dz[tt, kk][:, None] * uv[tt]).sum(axis=0)
    out.du, out.dg, out.dz, out.de = du, dg, dz, de
    if stack:
        def full(parts, shape):
            return np.stack([parts[e] if e in parts else np.zeros(shape) for e in range(N + 1)])
        out.dw1, out.dw3, out.dw2 = full(dW1, (I, d)), full(dW3, (I, d)), full(dW2, (d, I))
    else:
        out.dw1, out.dw3, out.dw2 = dW1, dW3, dW2
    return out


def sgd_f32(w, grad, lr) -> np.ndarray:
    """Plain SGD on an fp32 master: fl32(w - fl32(lr * fl32(grad)))."""
    step = (np.float32(lr) * _r32(grad)).astype(np.float32)
    return (np.asarray(w, np.float32) - step).astype(np.float32)


def train_step(u_bf16, masters: dict, bias: np.ndarray, K: int, G_bf16, lr: float, gamma: float, n_groups=1,
               topk_groups=1):
    """One training step of the layer (readings in moe_oracle.c, [train], [bias]):
    the FP8 forward and backward from the fp32 master weights (quantised per
    128x128 block), plain SGD w <- w - lr * dw on every master in fp32
    (fl32(w - fl32(lr * dw))), then the load-based bias update.

    masters: {"w1": [N+1, I, d], "w3": [N+1, I, d], "w2": [N+1, d, I],
    "e": [N, d]} fp32 arrays. Returns (new masters, new bias, Backward)."""
    m = {k: np.asarray(v, np.float32) for k, v in masters.items()}
    bw = layer_backward(u_bf16, m["e"], bias, K, lambda e: (m["w1"][e], m["w3"][e], m["w2"][e]), G_bf16,
                        n_groups=n_groups, topk_groups=topk_groups, fp8=True)
    new = {k: sgd_f32(m[k], grad, lr) for k, grad in (("w1", bw.dw1), ("w3", bw.dw3), ("w2", bw.dw2), ("e", bw.de))}
    T = as_bf16_bits(u_bf16).shape[0]
    new_bias = bias_update(bias, bw.route.loads, T, K, gamma)
    return new, new_bias, bw
