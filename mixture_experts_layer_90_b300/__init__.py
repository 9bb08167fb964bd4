"""Python binding of the B300 DeepSeekMoE layer-forward library (libmoe.so).

Argument marshalling only: every function passes torch tensors' device
pointers and the current CUDA stream to the C ABI declared in include/moe.h,
where every step of the computation runs in this package's CUDA kernels.
There is no fallback: importing works without a GPU, but any call raises if
the library is missing or no CUDA device is present.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_WORKSPACE, \
    MOE_ERR_DEVICE_DATA = range(7)
MOE_DTYPE_BF16, MOE_DTYPE_F32, MOE_DTYPE_E4M3 = 0, 1, 2
MOE_DISPATCH_SCATTER, MOE_DISPATCH_GATHER = 0, 1
MOE_EPI_BF16, MOE_EPI_SWIGLU_FP8, MOE_EPI_SWIGLU_BF16, MOE_EPI_F32 = 0, 1, 2, 3

EXPORTS = [
    "moe_last_error", "moe_num_sms", "moe_get_device_status",
    "fp8_quant_1x128", "fp8_quant_128x128",
    "moe_route_workspace_size", "moe_route",
    "moe_route_prepared_centroids_size", "moe_route_prepare_centroids",
    "moe_route_prepared_workspace_size", "moe_route_prepared",
    "moe_route_balance_stats_workspace_size", "moe_route_balance_stats",
    "moe_layer_train_workspace_size", "moe_layer_forward_train", "moe_layer_backward", "moe_layer_train_step",
    "moe_layer_train_buffer", "fp8_grouped_gemm_wgrad", "fp8_transpose_128x128", "moe_sgd_requant_128x128",
    "moe_sgd_f32",
    "moe_permute_workspace_size", "moe_permute", "moe_permute_static",
    "fp8_grouped_gemm", "bf16_grouped_gemm",
    "moe_combine", "moe_bias_update", "moe_selftest_wait_timeout",
    "moe_layer_workspace_size", "moe_layer_forward",
    "moe_layer_host_workspace_size", "moe_layer_forward_host",
    "moe_layer_host_pipeline_workspace_size", "moe_layer_forward_host_pipelined",
]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where} failed with status {status}: {text}")
        self.status = status


class LayerWeights(ctypes.Structure):
    """Mirror of moe_layer_weights."""
    _fields_ = [
        ("d", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int), ("I", ctypes.c_int),
        ("n_groups", ctypes.c_int), ("topk_groups", ctypes.c_int), ("gamma", ctypes.c_float),
        ("fp8", ctypes.c_int), ("centroids", ctypes.c_void_p), ("centroid_dtype", ctypes.c_int),
        ("bias", ctypes.c_void_p), ("w13", ctypes.c_void_p), ("w13_scales", ctypes.c_void_p),
        ("w2", ctypes.c_void_p), ("w2_scales", ctypes.c_void_p), ("centroids_prepared", ctypes.c_void_p),
        ("dispatch", ctypes.c_int),
    ]


class LayerWeightsT(ctypes.Structure):
    """moe_layer_weights_t: W13 and W2 quantised per 128x128 block, transposed."""
    _fields_ = [("w13t", ctypes.c_void_p), ("w13t_scales", ctypes.c_void_p), ("w2t", ctypes.c_void_p),
                ("w2t_scales", ctypes.c_void_p)]


class LayerGrads(ctypes.Structure):
    _fields_ = [("dw13", ctypes.c_void_p), ("dw2", ctypes.c_void_p), ("dcentroids", ctypes.c_void_p),
                ("dz", ctypes.c_void_p), ("stage_events", ctypes.c_void_p)]


BACKWARD_STAGES = 8


class LayerMasters(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p)]


TRAIN_BUFFERS = {"H": 0, "scores": 1, "dg": 2, "dA": 3, "dH": 4, "dX": 5, "offsets": 6, "perm_token": 7,
                 "dest_row": 8, "y": 9, "kofs": 10, "dy_q": 11, "dy_s": 12, "dh_q": 13, "dh_s": 14, "row_gate": 15, "logits": 16}


class LayerOutputs(ctypes.Structure):
    """Mirror of moe_layer_outputs."""
    _fields_ = [("topk_idx", ctypes.c_void_p), ("gates", ctypes.c_void_p), ("loads", ctypes.c_void_p),
                ("stage_events", ctypes.c_void_p)]


LAYER_STAGES = ("route", "permute", "gemm1_swiglu", "gemm2", "combine", "bias_update")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmoe.so (built by mixture_experts_layer_90_b300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mixture_experts_layer_90_b300.build`")
    L = ctypes.CDLL(path)
    i64, i32, vp, sz, flt = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    sig = {
        "moe_last_error": (ctypes.c_char_p, []),
        "moe_num_sms": (i32, []),
        "moe_get_device_status": (i32, [vp, ctypes.POINTER(ctypes.c_int)]),
        "fp8_quant_1x128": (i32, [vp, i64, i64, i64, vp, vp, i64, vp]),
        "fp8_quant_128x128": (i32, [vp, i64, i64, vp, vp, vp]),
        "moe_route_workspace_size": (sz, [i64, i32, i32, i32]),
        "moe_route": (i32, [vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
        "moe_route_prepared_centroids_size": (sz, [i32, i32, i32]),
        "moe_route_prepare_centroids": (i32, [vp, i32, i32, i32, vp, sz, vp]),
        "moe_route_prepared_workspace_size": (sz, [i64, i32, i32, i32]),
        "moe_route_prepared": (i32, [vp, i64, i32, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]),
        "moe_route_balance_stats_workspace_size": (sz, [i64, i32, i64]),
        "moe_route_balance_stats": (i32, [vp, vp, i64, i32, i32, i64, vp, vp, vp, vp, sz, vp]),
        "moe_permute_workspace_size": (sz, [i64, i32]),
        "moe_permute": (i32, [vp, i64, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_permute_static": (i32, [vp, i64, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
        "fp8_grouped_gemm": (i32, [vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, vp, vp]),
        "bf16_grouped_gemm": (i32, [vp, vp, vp, i32, i64, i32, i32, i32, vp, vp]),
        "moe_combine": (i32, [vp, vp, vp, vp, vp, i64, i32, i32, i64, vp, vp]),
        "moe_bias_update": (i32, [vp, vp, i32, i64, i32, flt, vp]),
        "moe_selftest_wait_timeout": (i32, [i64, vp]),
        "moe_layer_workspace_size": (sz, [ctypes.POINTER(LayerWeights), i64]),
        "moe_layer_forward": (i32, [ctypes.POINTER(LayerWeights), vp, i64, vp, ctypes.POINTER(LayerOutputs),
                                    i32, vp, sz, vp]),
        "moe_layer_host_workspace_size": (sz, [ctypes.POINTER(LayerWeights), i64]),
        "moe_layer_forward_host": (i32, [ctypes.POINTER(LayerWeights), vp, i64, vp,
                                         ctypes.POINTER(LayerOutputs), i32, vp, sz, vp]),
        "moe_layer_host_pipeline_workspace_size": (sz, [ctypes.POINTER(LayerWeights), i64]),
        "moe_layer_train_workspace_size": (sz, [ctypes.POINTER(LayerWeights), i64]),
        "moe_layer_forward_train": (i32, [ctypes.POINTER(LayerWeights), vp, i64, vp, ctypes.POINTER(LayerOutputs),
                                          i32, vp, sz, vp]),
        "moe_layer_backward": (i32, [ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerWeightsT), vp, i64, vp, vp,
                                     ctypes.POINTER(LayerGrads), vp, sz, vp]),
        "moe_layer_train_step": (i32, [ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerWeightsT),
                                       ctypes.POINTER(LayerMasters), vp, i64, vp, flt, vp, vp,
                                       ctypes.POINTER(LayerOutputs), ctypes.POINTER(LayerGrads), vp, sz, vp]),
        "moe_layer_train_buffer": (i32, [ctypes.POINTER(LayerWeights), i64, i32, ctypes.POINTER(sz),
                                         ctypes.POINTER(sz)]),
        "fp8_grouped_gemm_wgrad": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i64, vp, vp]),
        "fp8_transpose_128x128": (i32, [vp, vp, i32, i32, i32, vp, vp, vp]),
        "moe_sgd_requant_128x128": (i32, [vp, vp, i32, i32, i32, flt, vp, vp, vp, vp, vp]),
        "moe_sgd_f32": (i32, [vp, vp, i64, flt, vp]),
        "moe_layer_forward_host_pipelined": (i32, [ctypes.POINTER(LayerWeights), vp, i64, vp,
                                                   ctypes.POINTER(LayerOutputs), i32, i32, vp, sz, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _require_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: this library has no CPU path")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where, load_library().moe_last_error().decode())


def _ws(nbytes: int, device) -> torch.Tensor:
    # 256-byte aligned by torch's caching allocator (allocations are 512-byte aligned)
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def device_status() -> int:
    """Synchronises the current stream; returns and clears the device status word."""
    _require_cuda()
    v = ctypes.c_int(0)
    _check(load_library().moe_get_device_status(_stream(), ctypes.byref(v)), "moe_get_device_status")
    return v.value


# --------------------------------------------------------------------------
# one function per C entry point
# --------------------------------------------------------------------------

def fp8_quant_1x128(x: torch.Tensor, q: torch.Tensor = None, scales: torch.Tensor = None, ld_s: int = None):
    """bf16 [R, C] -> (e4m3 codes uint8 [R, C], scales fp32 [C/128, ld_s])."""
    _require_cuda()
    R, C = x.shape
    ld_s = R if ld_s is None else ld_s
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device) if q is None else q
    scales = torch.empty((C // 128, ld_s), dtype=torch.float32, device=x.device) if scales is None else scales
    _check(load_library().fp8_quant_1x128(_p(x), R, C, x.stride(0), _p(q), _p(scales), ld_s, _stream()),
           "fp8_quant_1x128")
    return q, scales


def fp8_quant_128x128(w: torch.Tensor, q: torch.Tensor = None, scales: torch.Tensor = None):
    """bf16 [R, C] -> (e4m3 codes uint8 [R, C], scales fp32 [ceil(R/128), C/128])."""
    _require_cuda()
    R, C = w.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=w.device) if q is None else q
    scales = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=w.device) if scales is None else scales
    _check(load_library().fp8_quant_128x128(_p(w), R, C, _p(q), _p(scales), _stream()), "fp8_quant_128x128")
    return q, scales


def moe_route(u, centroids, bias, K, n_groups=1, topk_groups=1, want_scores=False, workspace=None):
    """-> (topk_idx int32 [T,K], gates fp32 [T,K], loads int32 [N], scores fp32 [T,N] or None)."""
    _require_cuda()
    L = load_library()
    T, d = u.shape
    N = centroids.shape[0]
    cdt = MOE_DTYPE_F32 if centroids.dtype == torch.float32 else MOE_DTYPE_BF16
    dev = u.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    gates = torch.empty((T, K), dtype=torch.float32, device=dev)
    loads = torch.empty((N,), dtype=torch.int32, device=dev)
    scores = torch.empty((T, N), dtype=torch.float32, device=dev) if want_scores else None
    need = L.moe_route_workspace_size(T, d, N, cdt)
    ws = _ws(need, dev) if workspace is None else workspace
    _check(L.moe_route(_p(u), T, d, _p(centroids), cdt, _p(bias), N, K, n_groups, topk_groups, _p(idx), _p(gates),
                       _p(loads), _p(scores), _p(ws), ws.numel(), _stream()), "moe_route")
    return idx, gates, loads, scores


def moe_route_prepare_centroids(centroids, prepared=None):
    """-> the gate's tensor-core operand for these centroids (uint8 device buffer),
    to pass to moe_route_prepared while the centroids stay the same."""
    _require_cuda()
    L = load_library()
    N, d = centroids.shape
    cdt = MOE_DTYPE_F32 if centroids.dtype == torch.float32 else MOE_DTYPE_BF16
    need = L.moe_route_prepared_centroids_size(d, N, cdt)
    prepared = _ws(need, centroids.device) if prepared is None else prepared
    _check(L.moe_route_prepare_centroids(_p(centroids), cdt, N, d, _p(prepared), prepared.numel(), _stream()),
           "moe_route_prepare_centroids")
    return prepared


def moe_route_prepared(u, prepared, centroid_dtype, N, bias, K, n_groups=1, topk_groups=1, want_scores=False,
                       workspace=None):
    """moe_route from prepared centroids (centroid_dtype: MOE_DTYPE_F32 / MOE_DTYPE_BF16 of the
    centroids they came from) -> (topk_idx, gates, loads, scores or None)."""
    _require_cuda()
    L = load_library()
    T, d = u.shape
    dev = u.device
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    gates = torch.empty((T, K), dtype=torch.float32, device=dev)
    loads = torch.empty((N,), dtype=torch.int32, device=dev)
    scores = torch.empty((T, N), dtype=torch.float32, device=dev) if want_scores else None
    need = L.moe_route_prepared_workspace_size(T, d, N, centroid_dtype)
    ws = _ws(need, dev) if workspace is None else workspace
    _check(L.moe_route_prepared(_p(u), T, d, _p(prepared), centroid_dtype, _p(bias), N, K, n_groups, topk_groups,
                                _p(idx), _p(gates), _p(loads), _p(scores), _p(ws), ws.numel(), _stream()),
           "moe_route_prepared")
    return idx, gates, loads, scores


def moe_route_balance_stats(scores, topk_idx, seq_len, workspace=None):
    """Sequence-wise balance statistics (include/moe.h) from moe_route's scores
    [T, N] and topk_idx [T, K] -> (seq_loads int32 [S, N], seq_prob fp32 [S, N],
    seq_stat fp32 [S]), S = ceil(T / seq_len)."""
    _require_cuda()
    L = load_library()
    T, N = scores.shape
    K = topk_idx.shape[1]
    dev = scores.device
    S = (T + seq_len - 1) // seq_len
    loads = torch.empty((S, N), dtype=torch.int32, device=dev)
    prob = torch.empty((S, N), dtype=torch.float32, device=dev)
    stat = torch.empty((S,), dtype=torch.float32, device=dev)
    need = L.moe_route_balance_stats_workspace_size(T, N, seq_len)
    ws = _ws(need, dev) if workspace is None else workspace
    _check(L.moe_route_balance_stats(_p(scores), _p(topk_idx), T, N, K, seq_len, _p(loads), _p(prob), _p(stat),
                                     _p(ws), ws.numel(), _stream()), "moe_route_balance_stats")
    return loads, prob, stat


def moe_permute(x, topk_idx, N, out_dtype=MOE_DTYPE_BF16, with_shared=False, workspace=None):
    """-> (offsets int32 [N+1(+1)], perm_token int32 [T*K], dest_row int32 [T,K],
    x_perm [R, d] bf16 or uint8, x_perm_scales fp32 [d/128, R] or None)."""
    _require_cuda()
    L = load_library()
    T, d = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    R = T * K + (T if with_shared else 0)
    offsets = torch.empty((N + 1 + (1 if with_shared else 0),), dtype=torch.int32, device=dev)
    perm = torch.empty((T * K,), dtype=torch.int32, device=dev)
    dest = torch.empty((T, K), dtype=torch.int32, device=dev)
    fp8 = out_dtype == MOE_DTYPE_E4M3
    xp = torch.empty((R, d), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xs = torch.empty((d // 128, R), dtype=torch.float32, device=dev) if fp8 else None
    need = L.moe_permute_workspace_size(T, N)
    ws = _ws(need, dev) if workspace is None else workspace
    _check(L.moe_permute(_p(x), T, d, _p(topk_idx), N, K, out_dtype, int(bool(with_shared)), _p(offsets), _p(perm),
                         _p(dest), _p(xp), _p(xs), _p(ws), ws.numel(), _stream()), "moe_permute")
    return offsets, perm, dest, xp, xs


def moe_permute_static(x, topk_idx, N, out_dtype=MOE_DTYPE_BF16, with_shared=False):
    """moe_permute without a workspace: its scratch is a fixed array inside the
    library (for callers that cannot allocate device memory). Same outputs."""
    _require_cuda()
    L = load_library()
    T, d = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    R = T * K + (T if with_shared else 0)
    offsets = torch.empty((N + 1 + (1 if with_shared else 0),), dtype=torch.int32, device=dev)
    perm = torch.empty((T * K,), dtype=torch.int32, device=dev)
    dest = torch.empty((T, K), dtype=torch.int32, device=dev)
    fp8 = out_dtype == MOE_DTYPE_E4M3
    xp = torch.empty((R, d), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xs = torch.empty((d // 128, R), dtype=torch.float32, device=dev) if fp8 else None
    _check(L.moe_permute_static(_p(x), T, d, _p(topk_idx), N, K, out_dtype, int(bool(with_shared)), _p(offsets),
                                _p(perm), _p(dest), _p(xp), _p(xs), _stream()), "moe_permute_static")
    return offsets, perm, dest, xp, xs


def fp8_grouped_gemm(A, sa, B, sb, group_offsets, epilogue=MOE_EPI_BF16, C=None, c_scales=None):
    """A uint8 [M, Kd], sa fp32 [Kd/128, M], B uint8 [G, Nd, Kd], sb fp32 [G, Nd/128, Kd/128],
    group_offsets int32 [G+1] -> C (bf16 [M, Nd], or e4m3 [M, Nd/2] + scales [Nd/256, M])."""
    _require_cuda()
    M, Kd = A.shape
    G, Nd, _ = B.shape
    dev = A.device
    if C is None:
        if epilogue == MOE_EPI_SWIGLU_FP8:
            C = torch.empty((M, Nd // 2), dtype=torch.uint8, device=dev)
            c_scales = torch.empty((Nd // 256, M), dtype=torch.float32, device=dev)
        else:
            C = torch.empty((M, Nd), dtype=torch.bfloat16, device=dev)
    _check(load_library().fp8_grouped_gemm(_p(A), _p(sa), _p(B), _p(sb), _p(group_offsets), G, M, Nd, Kd, epilogue,
                                           _p(C), _p(c_scales), _stream()), "fp8_grouped_gemm")
    return (C, c_scales) if epilogue == MOE_EPI_SWIGLU_FP8 else C


def bf16_grouped_gemm(A, B, group_offsets, epilogue=MOE_EPI_BF16, C=None):
    """A bf16 [M, Kd], B bf16 [G, Nd, Kd] -> C bf16 [M, Nd] / [M, Nd/2] or fp32 [M, Nd]."""
    _require_cuda()
    M, Kd = A.shape
    G, Nd, _ = B.shape
    if C is None:
        if epilogue == MOE_EPI_F32:
            C = torch.empty((M, Nd), dtype=torch.float32, device=A.device)
        else:
            C = torch.empty((M, Nd // 2 if epilogue == MOE_EPI_SWIGLU_BF16 else Nd), dtype=torch.bfloat16,
                            device=A.device)
    _check(load_library().bf16_grouped_gemm(_p(A), _p(B), _p(group_offsets), G, M, Nd, Kd, epilogue, _p(C),
                                            _stream()), "bf16_grouped_gemm")
    return C


def moe_combine(u, y_shared, y_perm, gates, dest_row, out=None):
    """h' = u + y_shared + sum_k gates[:,k] * y_perm[dest_row[:,k]] (bf16 [T, d])."""
    _require_cuda()
    T, d = u.shape
    K = gates.shape[1]
    out = torch.empty_like(u) if out is None else out
    _check(load_library().moe_combine(_p(u), _p(y_shared), _p(y_perm), _p(gates), _p(dest_row), T, d, K,
                                      y_perm.shape[0], _p(out), _stream()), "moe_combine")
    return out


def moe_selftest_wait_timeout(limit_ns: int):
    """Launches a bounded wait that must time out (see include/moe.h)."""
    _require_cuda()
    _check(load_library().moe_selftest_wait_timeout(int(limit_ns), _stream()), "moe_selftest_wait_timeout")


def moe_bias_update(bias, loads, T, K, gamma):
    """In place: bias -= gamma where load > T*K/N, += gamma where below."""
    _require_cuda()
    _check(load_library().moe_bias_update(_p(bias), _p(loads), bias.numel(), T, K, float(gamma), _stream()),
           "moe_bias_update")
    return bias


# --------------------------------------------------------------------------
# training (include/moe.h, "Training")
# --------------------------------------------------------------------------

def fp8_grouped_gemm_wgrad(A, sa, B, sb, kofs, out=None):
    """FP8 weight-gradient GEMM grouped along K: A e4m3 [M, Kp], sa [Kp/128, M],
    B e4m3 [Nd, Kp], sb [Kp/128, Nd], kofs int32 [G+1] (device, 128-K block
    offsets of the groups) -> C fp32 [G, M, Nd]."""
    _require_cuda()
    M, Kp = A.shape
    Nd = B.shape[0]
    G = kofs.numel() - 1
    out = torch.empty((G, M, Nd), dtype=torch.float32, device=A.device) if out is None else out
    _check(load_library().fp8_grouped_gemm_wgrad(_p(A), _p(sa), _p(B), _p(sb), _p(kofs), G, M, Nd, Kp, _p(out),
                                                 _stream()), "fp8_grouped_gemm_wgrad")
    return out


def fp8_transpose_128x128(q, s, qt=None, st=None):
    """E4M3 codes [G, rows, cols] and 128x128 scales [G, rows/128, cols/128] ->
    (codes [G, cols, rows], scales [G, cols/128, rows/128])."""
    _require_cuda()
    G, rows, cols = q.shape
    qt = torch.empty((G, cols, rows), dtype=torch.uint8, device=q.device) if qt is None else qt
    st = torch.empty((G, cols // 128, rows // 128), dtype=torch.float32, device=q.device) if st is None else st
    _check(load_library().fp8_transpose_128x128(_p(q), _p(s), G, rows, cols, _p(qt), _p(st), _stream()),
           "fp8_transpose_128x128")
    return qt, st


def moe_sgd_requant_128x128(w, grad, lr, q, s, qt, st):
    """w [G, rows, cols] fp32 <- fl32(w - fl32(lr grad)); then q, s (128x128
    E4M3 and scales of the new w) and qt, st (the same, transposed)."""
    _require_cuda()
    G, rows, cols = w.shape
    _check(load_library().moe_sgd_requant_128x128(_p(w), _p(grad), G, rows, cols, float(lr), _p(q), _p(s), _p(qt),
                                                   _p(st), _stream()), "moe_sgd_requant_128x128")


def moe_sgd_f32(w, grad, lr):
    _require_cuda()
    _check(load_library().moe_sgd_f32(_p(w), _p(grad), w.numel(), float(lr), _stream()), "moe_sgd_f32")


from .layer import MoELayer  # noqa: E402  (after the entry points it wraps)
