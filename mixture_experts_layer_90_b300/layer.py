"""MoELayer: device-resident weights of one DeepSeekMoE layer and its forward.

The layer formula (nlp-lineage.vercel.app "DeepSeek-V3 Technical Report
(2024)", "The notation"): h'_t = u_t + FFN_shared(u_t) + sum_i g_{i,t} FFN_i(u_t),
one shared expert and N routed experts (top-K), every FFN a SwiGLU MLP whose
weights live in HBM as E4M3 with 128x128 block scales (or bf16).

Layout (all device memory, allocated once here, never by the C library):
  w13 [N+1, 2I, d]  gate and up projections, rows interleaved per 128
                    (gate rows 128j.., then up rows 128j..), expert N = shared
  w2  [N+1, d, I]   down projections
  *_scales          fp32 [N+1, rows/128, cols/128]

Training (FP8 layers; enable_training or build(..., train=True)) adds fp32
masters of w13 and w2, their FP8 codes transposed per 128x128 block (w13t
[N+1, d, 2I], w2t [N+1, I, d], for the backward's products) and the
gradients dw13, dw2 (fp32, the masters' layouts) and dcentroids [N, d].
"""
from __future__ import annotations

import ctypes

import torch

from . import (MOE_DISPATCH_GATHER, MOE_DISPATCH_SCATTER, MOE_DTYPE_BF16, MOE_DTYPE_F32, TRAIN_BUFFERS, LayerGrads, LayerMasters, LayerOutputs, LayerWeights,
               LayerWeightsT, _check, _p, _require_cuda, _stream, fp8_quant_128x128, fp8_transpose_128x128,
               load_library, moe_route_prepare_centroids)


def interleave_gate_up(w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    """[I, d] gate and [I, d] up -> [2I, d] with 128-row blocks alternating."""
    I, d = w1.shape
    return torch.stack((w1.view(I // 128, 128, d), w3.view(I // 128, 128, d)), dim=1).reshape(2 * I, d)


class MoELayer:
    def __init__(self, d, N, K, I, centroids, bias, w13, w2, w13_scales=None, w2_scales=None, n_groups=1,
                 topk_groups=1, gamma=1e-3, dispatch="scatter"):
        """dispatch (FP8 layers): "scatter" (the permutation writes the grouped rows) or
        "gather" (GEMM 1 gathers the quantised tokens by perm_token); the same bits."""
        _require_cuda()
        modes = {"scatter": MOE_DISPATCH_SCATTER, "gather": MOE_DISPATCH_GATHER}
        if dispatch not in modes:
            raise ValueError(f"dispatch must be one of {sorted(modes)}, not {dispatch!r}")
        self.d, self.N, self.K, self.I = d, N, K, I
        self.n_groups, self.topk_groups, self.gamma = n_groups, topk_groups, gamma
        self.fp8 = w13.dtype == torch.uint8
        self.centroids, self.bias = centroids, bias
        self.w13, self.w2, self.w13_scales, self.w2_scales = w13, w2, w13_scales, w2_scales
        # the gate's operand is prepared once: the centroids stay fixed, only the bias moves
        self.centroids_prepared = moe_route_prepare_centroids(centroids)
        self._desc = LayerWeights(
            d=d, N=N, K=K, I=I, n_groups=n_groups, topk_groups=topk_groups, gamma=gamma, fp8=int(self.fp8),
            centroids=centroids.data_ptr(),
            centroid_dtype=MOE_DTYPE_F32 if centroids.dtype == torch.float32 else MOE_DTYPE_BF16,
            bias=bias.data_ptr(), w13=w13.data_ptr(),
            w13_scales=w13_scales.data_ptr() if w13_scales is not None else None,
            w2=w2.data_ptr(), w2_scales=w2_scales.data_ptr() if w2_scales is not None else None,
            centroids_prepared=self.centroids_prepared.data_ptr(),
            dispatch=modes[dispatch])
        self._ws = {}
        self.loads = torch.zeros((N,), dtype=torch.int32, device=centroids.device)

    @classmethod
    def build(cls, d, N, K, I, centroids, bias, expert_weights, fp8=True, train=False, **kw):
        """expert_weights(e) -> (w1 [I,d], w3 [I,d], w2 [d,I]) bf16 device tensors for
        e in 0..N (N = shared expert); quantised here per 128x128 block when fp8.
        train: also keep fp32 masters of the weights and set up training."""
        dev = centroids.device
        G = N + 1
        if train:
            w13m = torch.empty((G, 2 * I, d), dtype=torch.float32, device=dev)
            w2m = torch.empty((G, d, I), dtype=torch.float32, device=dev)
        if fp8:
            w13 = torch.empty((G, 2 * I, d), dtype=torch.uint8, device=dev)
            w2 = torch.empty((G, d, I), dtype=torch.uint8, device=dev)
            s13 = torch.empty((G, 2 * I // 128, d // 128), dtype=torch.float32, device=dev)
            s2 = torch.empty((G, d // 128, I // 128), dtype=torch.float32, device=dev)
        else:
            w13 = torch.empty((G, 2 * I, d), dtype=torch.bfloat16, device=dev)
            w2 = torch.empty((G, d, I), dtype=torch.bfloat16, device=dev)
            s13 = s2 = None
        for e in range(G):
            w1, w3, w2e = expert_weights(e)
            w13e = interleave_gate_up(w1, w3)
            if train:
                w13m[e].copy_(w13e)
                w2m[e].copy_(w2e)
            if fp8:
                fp8_quant_128x128(w13e, w13[e], s13[e])
                fp8_quant_128x128(w2e.contiguous(), w2[e], s2[e])
            else:
                w13[e].copy_(w13e)
                w2[e].copy_(w2e)
        layer = cls(d, N, K, I, centroids, bias, w13, w2, s13, s2, **kw)
        if train:
            layer.enable_training(w13m, w2m)
        return layer

    def prepare_centroids(self):
        """Re-prepares the gate's operand; call after changing self.centroids in place."""
        moe_route_prepare_centroids(self.centroids, self.centroids_prepared)

    def workspace(self, T: int, host=False) -> torch.Tensor:
        """host: False (device buffers), True (host-buffer call) or "pipeline"."""
        key = (T, host)
        ws = self._ws.get(key)
        if ws is None:
            L = load_library()
            f = (L.moe_layer_host_pipeline_workspace_size if host == "pipeline" else
                 L.moe_layer_host_workspace_size if host else L.moe_layer_workspace_size)
            need = f(ctypes.byref(self._desc), T)
            ws = torch.empty((max(int(need), 1),), dtype=torch.uint8, device=self.centroids.device)
            self._ws[key] = ws
        return ws

    def _outs(self, topk_idx, gates, events=None):
        self._ev_arr = None
        if events is not None:
            for e in events:
                if e.cuda_event == 0:      # torch creates the CUDA event on its first record
                    e.record()
            self._ev_arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        return LayerOutputs(topk_idx=topk_idx.data_ptr() if topk_idx is not None else None,
                            gates=gates.data_ptr() if gates is not None else None,
                            loads=self.loads.data_ptr(),
                            stage_events=ctypes.cast(self._ev_arr, ctypes.c_void_p) if events is not None else None)

    def forward(self, u: torch.Tensor, out: torch.Tensor = None, update_bias: bool = True, topk_idx=None,
                gates=None, stage_events=None) -> torch.Tensor:
        """u bf16 [T, d] on the device -> h' bf16 [T, d]; then the bias update.
        stage_events: optional 7 torch.cuda.Event(enable_timing=True) recorded
        around the six stages on the current stream."""
        T = u.shape[0]
        out = torch.empty_like(u) if out is None else out
        ws = self.workspace(T)
        outs = self._outs(topk_idx, gates, stage_events)
        _check(load_library().moe_layer_forward(ctypes.byref(self._desc), _p(u), T, _p(out), ctypes.byref(outs),
                                                int(update_bias), _p(ws), ws.numel(), _stream()),
               "moe_layer_forward")
        return out

    def capture(self, u: torch.Tensor, out: torch.Tensor = None, update_bias: bool = True) -> "LayerGraph":
        """Records one forward on the static buffers u -> out into a CUDA graph
        (the library's calls are asynchronous, allocate nothing and never
        synchronise, so the whole launch sequence can be captured). Replaying it
        runs the layer on whatever u holds at replay time, writing out, the loads
        and, with update_bias, the bias. One eager call runs first, outside the
        capture, so that per-device set-up is done before it. The graph uses
        this layer's weights and its cached workspace for u's row count: the
        LayerGraph holds the layer, so they outlive it."""
        out = torch.empty_like(u) if out is None else out
        self.forward(u, out, update_bias=False)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(u, out, update_bias=update_bias)
        return LayerGraph(g, u, out, self)

    def forward_host(self, u_host: torch.Tensor, out_host: torch.Tensor, update_bias: bool = True):
        """Same with u/h' in (pinned) host memory: copies in and out inside the call."""
        T = u_host.shape[0]
        ws = self.workspace(T, host=True)
        outs = self._outs(None, None)
        _check(load_library().moe_layer_forward_host(ctypes.byref(self._desc), ctypes.c_void_p(u_host.data_ptr()), T,
                                                     ctypes.c_void_p(out_host.data_ptr()), ctypes.byref(outs),
                                                     int(update_bias), _p(ws), ws.numel(), _stream()),
               "moe_layer_forward_host")
        return out_host

    def forward_host_pipelined(self, u_host: torch.Tensor, out_host: torch.Tensor, slot: int,
                               done: torch.cuda.Event, update_bias: bool = True):
        """Pipelined host-buffer forward: alternate slot 0/1 between consecutive
        calls; `done` (an Event) completes once out_host holds h'."""
        T = u_host.shape[0]
        ws = self.workspace(T, host="pipeline")
        outs = self._outs(None, None)
        if done.cuda_event == 0:        # torch creates the CUDA event on its first record
            done.record()
        _check(load_library().moe_layer_forward_host_pipelined(
            ctypes.byref(self._desc), ctypes.c_void_p(u_host.data_ptr()), T, ctypes.c_void_p(out_host.data_ptr()),
            ctypes.byref(outs), int(update_bias), int(slot), _p(ws), ws.numel(), _stream(),
            ctypes.c_void_p(done.cuda_event)), "moe_layer_forward_host_pipelined")
        return out_host

    # ------------------------------------------------------------------
    # training
    # ------------------------------------------------------------------

    def enable_training(self, w13_master: torch.Tensor, w2_master: torch.Tensor):
        """fp32 masters [N+1, 2I, d] (W13's interleaved rows) and [N+1, d, I]
        whose 128x128 quantisation the layer's FP8 weights are; allocates the
        transposed FP8 weights and the gradients."""
        if not self.fp8:
            raise ValueError("training needs a FP8 layer")
        dev, G, d, I, N = self.centroids.device, self.N + 1, self.d, self.I, self.N
        self.w13_master, self.w2_master = w13_master, w2_master
        self.w13t, self.w13t_scales = fp8_transpose_128x128(self.w13, self.w13_scales)
        self.w2t, self.w2t_scales = fp8_transpose_128x128(self.w2, self.w2_scales)
        self.dw13 = torch.empty((G, 2 * I, d), dtype=torch.float32, device=dev)
        self.dw2 = torch.empty((G, d, I), dtype=torch.float32, device=dev)
        self.dcentroids = torch.empty((N, d), dtype=torch.float32, device=dev)
        self._wt = LayerWeightsT(w13t=self.w13t.data_ptr(), w13t_scales=self.w13t_scales.data_ptr(),
                                 w2t=self.w2t.data_ptr(), w2t_scales=self.w2t_scales.data_ptr())
        self._masters = LayerMasters(w13=w13_master.data_ptr(), w2=w2_master.data_ptr())
        self._train_ws = {}

    def train_workspace(self, T: int) -> torch.Tensor:
        ws = self._train_ws.get(T)
        if ws is None:
            need = load_library().moe_layer_train_workspace_size(ctypes.byref(self._desc), T)
            ws = torch.empty((max(int(need), 1),), dtype=torch.uint8, device=self.centroids.device)
            self._train_ws[T] = ws
        return ws

    def train_buffer(self, T: int, name: str) -> torch.Tensor:
        """A named buffer of the training workspace for T tokens (after
        forward_train / backward): H, scores, dg, dA, dH, dX, offsets,
        perm_token, dest_row, y, kofs, dy_q, dy_s, dh_q, dh_s, row_gate, logits."""
        off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        _check(load_library().moe_layer_train_buffer(ctypes.byref(self._desc), T, TRAIN_BUFFERS[name],
                                                     ctypes.byref(off), ctypes.byref(nb)), "moe_layer_train_buffer")
        raw = self.train_workspace(T)[off.value:off.value + nb.value]
        R, d, I, N, K = T * self.K + T, self.d, self.I, self.N, self.K
        shape, dtype = {
            "H": ((R, 2 * I), torch.bfloat16), "scores": ((T, N), torch.float32), "dg": ((T, K), torch.float32),
            "dA": ((R, I), torch.bfloat16), "dH": ((R, 2 * I), torch.bfloat16), "dX": ((R, d), torch.bfloat16),
            "offsets": ((N + 2,), torch.int32), "perm_token": ((T * K,), torch.int32),
            "dest_row": ((T, K), torch.int32), "y": ((R, d), torch.bfloat16), "kofs": ((N + 2,), torch.int32),
            "dy_q": ((R, d), torch.uint8), "dy_s": ((d // 128, R), torch.float32),
            "dh_q": ((R, 2 * I), torch.uint8), "dh_s": ((2 * I // 128, R), torch.float32),
            "row_gate": ((R,), torch.float32), "logits": ((T, N), torch.float32),
        }[name]
        return raw.view(dtype).view(shape)

    def _grads(self, dz, events=None):
        self._bwd_ev = None
        if events is not None:
            for e in events:
                if e.cuda_event == 0:      # torch creates the CUDA event on its first record
                    e.record()
            self._bwd_ev = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        return LayerGrads(dw13=self.dw13.data_ptr(), dw2=self.dw2.data_ptr(), dcentroids=self.dcentroids.data_ptr(),
                          dz=dz.data_ptr() if dz is not None else None,
                          stage_events=ctypes.cast(self._bwd_ev, ctypes.c_void_p) if events is not None else None)

    def forward_train(self, u: torch.Tensor, out: torch.Tensor = None, update_bias: bool = True, topk_idx=None,
                      gates=None) -> torch.Tensor:
        """forward that keeps what the backward reads (in the training workspace)."""
        T = u.shape[0]
        out = torch.empty_like(u) if out is None else out
        ws = self.train_workspace(T)
        outs = self._outs(topk_idx, gates)
        _check(load_library().moe_layer_forward_train(ctypes.byref(self._desc), _p(u), T, _p(out),
                                                      ctypes.byref(outs), int(update_bias), _p(ws), ws.numel(),
                                                      _stream()), "moe_layer_forward_train")
        return out

    def backward(self, u: torch.Tensor, dout: torch.Tensor, du: torch.Tensor = None, dz: torch.Tensor = None,
                 stage_events=None):
        """Gradients of the last forward_train on u: dout = dL/dh' bf16 [T, d] ->
        du bf16 [T, d]; dw13, dw2, dcentroids (and dz [T, K] if given) filled.
        stage_events: optional 9 torch.cuda.Event(enable_timing=True) recorded
        around the backward's eight stages on the current stream."""
        T = u.shape[0]
        du = torch.empty_like(u) if du is None else du
        ws = self.train_workspace(T)
        grads = self._grads(dz, stage_events)
        _check(load_library().moe_layer_backward(ctypes.byref(self._desc), ctypes.byref(self._wt), _p(u), T,
                                                 _p(dout), _p(du), ctypes.byref(grads), _p(ws), ws.numel(),
                                                 _stream()), "moe_layer_backward")
        return du

    def capture_train(self, u: torch.Tensor, dout: torch.Tensor, lr: float, out: torch.Tensor = None,
                      du: torch.Tensor = None) -> "TrainGraph":
        """Records one training step on the static buffers u, dout -> out, du
        into a CUDA graph (learning rate fixed at capture). A training forward
        and backward run first, outside the capture, with no update (no bias
        move, no SGD), so that per-device set-up and the workspace exist."""
        out = torch.empty_like(u) if out is None else out
        du = torch.empty_like(u) if du is None else du
        self.forward_train(u, out, update_bias=False)
        self.backward(u, dout, du)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.train_step(u, dout, lr, out, du)
        return TrainGraph(g, u, dout, out, du, self)

    def train_step(self, u: torch.Tensor, dout: torch.Tensor, lr: float, out: torch.Tensor = None,
                   du: torch.Tensor = None):
        """One SGD step (forward_train with the bias update, backward, SGD on the
        masters and the fp32 centroids, FP8 weights quantised again) -> (h', du)."""
        T = u.shape[0]
        out = torch.empty_like(u) if out is None else out
        du = torch.empty_like(u) if du is None else du
        ws = self.train_workspace(T)
        outs = self._outs(None, None)
        grads = self._grads(None)
        _check(load_library().moe_layer_train_step(ctypes.byref(self._desc), ctypes.byref(self._wt),
                                                   ctypes.byref(self._masters), _p(u), T, _p(dout), float(lr),
                                                   _p(out), _p(du), ctypes.byref(outs), ctypes.byref(grads), _p(ws),
                                                   ws.numel(), _stream()), "moe_layer_train_step")
        return out, du


class TrainGraph:
    """A captured training step: copy a batch into `u` and its dL/dh' into
    `dout`, call replay(); `out`, `du` and the layer's weights, bias and
    centroids then hold the step's results."""

    def __init__(self, graph, u, dout, out, du, layer):
        self.graph, self.u, self.dout, self.out, self.du, self.layer = graph, u, dout, out, du, layer

    def replay(self):
        self.graph.replay()
        return self.out, self.du


class LayerGraph:
    """A captured layer forward: copy a batch into `u`, call replay(), read `out`."""

    def __init__(self, graph, u, out, layer):
        self.graph, self.u, self.out, self.layer = graph, u, out, layer

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out
