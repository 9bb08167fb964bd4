"""The whole layer on the GPU (route, permute, grouped SwiGLU GEMMs with the
shared expert, combine, bias update) against the oracle's FP64 chain.

Layer formula: nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)",
"The notation". h' must be within the bf16-rounding rule of tests/helpers.py
at tau = 2e-3 (normwise per token); routing, loads and the bias bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import check_bf16

pytestmark = pytest.mark.gpu

from helpers import ROUTE_DELTA as DELTA


def _lib():
    import mixture_experts_layer_90_b300 as m
    return m


def _build(sh, zipf=False, zero_bias=False):
    m = _lib()
    cent = S.centroids(sh, zipf=zipf).cuda()
    bias = S.bias(sh, zero=zero_bias).cuda()
    layer = m.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias,
                             lambda e: S.expert_weights(sh, e, device="cuda"), fp8=sh.fp8,
                             n_groups=sh.n_groups, topk_groups=sh.topk_groups, gamma=sh.gamma)
    return layer


def _cpu_weights(sh):
    return lambda e: tuple(w.cpu() for w in S.expert_weights(sh, e, device="cuda"))


def _run_and_check(sh, tokens=None, zipf=False, zero_bias=False, u_seed=0, pick=None):
    """Runs the layer on the GPU, then checks routing, loads and the bias for all
    tokens and h' for `tokens` (all if None), or for pick(topk_idx, loads) when
    the tokens to check depend on the routing."""
    m = _lib()
    layer = _build(sh, zipf=zipf, zero_bias=zero_bias)
    b0 = layer.bias.cpu().numpy().copy()
    u = S.tokens(sh, seed=u_seed)
    T = sh.T
    idx = torch.empty((T, sh.K), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, sh.K), dtype=torch.float32, device="cuda")
    out = layer.forward(u.cuda(), topk_idx=idx, gates=gates, update_bias=True)
    assert m.device_status() == 0
    idx_g, loads_g = idx.cpu().numpy(), layer.loads.cpu().numpy()
    if pick is not None:
        tokens = pick(idx_g, loads_g)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    ref, r, _ = oracle.layer_tokens(u, layer.centroids.cpu(), torch.from_numpy(b0), sh.K, _cpu_weights(sh), tokens,
                                    fp8=sh.fp8, n_groups=sh.n_groups, topk_groups=sh.topk_groups, delta=DELTA)
    same = np.all(idx_g == r.topk_idx, axis=1)
    assert np.all(same | r.near_tie), "token with a certified gap routed differently"
    np.testing.assert_array_equal(loads_g, np.bincount(idx_g.ravel(), minlength=sh.N))
    if same.all():
        np.testing.assert_array_equal(loads_g, r.loads)
    # bias after the step: one fp32 step from this step's loads
    np.testing.assert_array_equal(layer.bias.cpu().numpy(), oracle.bias_update(b0, loads_g, T, sh.K, sh.gamma))
    keep = same[tokens]
    got = out[torch.as_tensor(tokens[keep]).cuda()].cpu()
    tau = check_bf16(got, ref[keep], tau=2e-3, what=sh.name)
    return tau, int((~same).sum())


def test_layer_tiny_bf16():
    """The tiny bf16 layer: T=128, d=256, 16 routed + 1 shared, top-4, I=128, b=0."""
    tau, _ = _run_and_check(S.TINY, zero_bias=True)
    assert tau < 2e-3


def test_layer_small_fp8_ragged():
    sh = S.LayerShape(T=301, d=512, N=32, K=4, I=256, name="small-fp8")
    _run_and_check(sh)


def test_layer_small_fp8_group_limited():
    sh = S.LayerShape(T=96, d=512, N=64, K=6, I=256, n_groups=8, topk_groups=3, name="small-fp8-groups")
    _run_and_check(sh)


def test_layer_second_step_uses_updated_bias():
    sh = S.LayerShape(T=128, d=256, N=16, K=4, I=128, name="two-steps")
    layer = _build(sh)
    u = S.tokens(sh).cuda()
    layer.forward(u)
    b1 = layer.bias.clone()
    l1 = layer.loads.clone()
    layer.forward(u)
    b_exp = oracle.bias_update(b1.cpu().numpy(), layer.loads.cpu().numpy(), sh.T, sh.K, sh.gamma)
    np.testing.assert_array_equal(layer.bias.cpu().numpy(), b_exp)
    assert not torch.equal(b1, S.bias(sh).cuda()) or l1.sum() == sh.T * sh.K


def test_layer_empty_batch():
    sh = S.LayerShape(T=0, d=256, N=16, K=4, I=128, name="empty")
    layer = _build(sh)
    b0 = layer.bias.clone()
    out = layer.forward(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, 256) and _lib().device_status() == 0
    # no tokens: every expert is underloaded only if the mean (0) exceeds its load, which never happens
    assert torch.equal(layer.bias, b0)


def test_layer_host_buffers_match_device_path():
    sh = S.LayerShape(T=200, d=512, N=32, K=4, I=256, name="host")
    layer = _build(sh)
    u = S.tokens(sh)
    out_d = layer.forward(u.cuda(), update_bias=False).cpu()
    u_h = u.pin_memory()
    out_h = torch.empty_like(u_h).pin_memory()
    layer.forward_host(u_h, out_h, update_bias=False)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16))


def test_layer_pipelined_host_calls_match_device_path():
    """Four consecutive pipelined host-buffer calls (slots 0,1,0,1, different
    batches) give exactly what the device-buffer call gives for each batch."""
    sh = S.LayerShape(T=160, d=512, N=32, K=4, I=256, name="pipe")
    layer = _build(sh)
    us = [S.tokens(sh, seed=10 + i) for i in range(4)]
    expect = [layer.forward(u.cuda(), update_bias=False).cpu() for u in us]
    u_h = [u.pin_memory() for u in us]
    out_h = [torch.empty_like(u).pin_memory() for u in us]
    done = [torch.cuda.Event() for _ in us]
    for i in range(4):
        layer.forward_host_pipelined(u_h[i], out_h[i], slot=i % 2, done=done[i], update_bias=False)
    for i in range(4):
        done[i].synchronize()
        assert torch.equal(out_h[i].view(torch.int16), expect[i].view(torch.int16)), i
    assert _lib().device_status() == 0


def test_layer_with_and_without_prepared_centroids_agree():
    """The layer routes from centroids prepared once at set-up; routing from the
    raw centroids inside the call gives the same bits."""
    sh = S.LayerShape(T=130, d=512, N=32, K=4, I=256, name="prepared")
    layer = _build(sh)
    u = S.tokens(sh).cuda()
    a = layer.forward(u, update_bias=False)
    layer._desc.centroids_prepared = None
    layer._ws.clear()
    b = layer.forward(u, update_bias=False)
    assert _lib().device_status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fp8", [False, True])
def test_layer_graph_replay_matches_eager(fp8):
    """The layer captured in a CUDA graph and replayed on new batches gives the
    same bits as the eager call: h', the loads and the bias after two updates."""
    sh = S.LayerShape(T=128, d=256, N=16, K=4, I=128, fp8=fp8, centroid_f32=fp8, name=f"graph-{fp8}")
    eager, graphed = _build(sh), _build(sh)
    u = torch.empty((sh.T, sh.d), dtype=torch.bfloat16, device="cuda")
    g = graphed.capture(u)
    for seed in (21, 22):
        batch = S.tokens(sh, seed=seed).cuda()
        ref = eager.forward(batch)
        u.copy_(batch)
        got = g.replay()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(graphed.loads, eager.loads)
        assert torch.equal(graphed.bias, eager.bias)
    assert _lib().device_status() == 0


@pytest.mark.parametrize("sh", [S.LayerShape(T=301, d=512, N=32, K=4, I=256, name="dispatch-ragged"),
                                S.LayerShape(T=96, d=512, N=64, K=6, I=256, n_groups=8, topk_groups=3,
                                             name="dispatch-groups"),
                                S.LayerShape(T=1, d=256, N=8, K=2, I=128, name="dispatch-one-token")])
def test_layer_gather_and_scatter_dispatch_agree(sh):
    """GEMM 1 gathering the quantised tokens by perm_token and the permutation
    writing the grouped rows (the default) give the same bits: h', the routing,
    the loads and the bias after an update."""
    m = _lib()
    layer = _build(sh)
    b0 = layer.bias.clone()
    u = S.tokens(sh).cuda()
    res = {}
    for mode in (m.MOE_DISPATCH_GATHER, m.MOE_DISPATCH_SCATTER):
        layer.bias.copy_(b0)
        layer._desc.dispatch = mode
        idx = torch.empty((sh.T, sh.K), dtype=torch.int32, device="cuda")
        gates = torch.empty((sh.T, sh.K), dtype=torch.float32, device="cuda")
        out = layer.forward(u, topk_idx=idx, gates=gates, update_bias=True)
        res[mode] = (out.clone(), idx, gates, layer.loads.clone(), layer.bias.clone())
        assert m.device_status() == 0
    for a, b in zip(res[m.MOE_DISPATCH_GATHER], res[m.MOE_DISPATCH_SCATTER]):
        assert torch.equal(_bits(a), _bits(b))


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16) if t.dtype == torch.bfloat16 \
        else t


def test_training_backward_same_under_both_dispatches():
    """The training forward keeps GEMM 1's products for the backward; with the
    gathered dispatch they, and so every gradient, are the scattered one's bits."""
    m = _lib()
    sh = S.LayerShape(T=300, d=256, N=8, K=2, I=256, name="dispatch-train")
    layer = m.MoELayer.build(sh.d, sh.N, sh.K, sh.I, S.centroids(sh).cuda(), S.bias(sh).cuda(),
                             lambda e: S.expert_weights(sh, e, device="cuda"), fp8=True, train=True, gamma=sh.gamma)
    u = S.tokens(sh, seed=3).cuda()
    G = S.grad_out(sh, seed=4).cuda()
    res = {}
    for mode in (m.MOE_DISPATCH_GATHER, m.MOE_DISPATCH_SCATTER):
        layer._desc.dispatch = mode
        out = layer.forward_train(u, update_bias=False)
        du = layer.backward(u, G)
        res[mode] = [out.clone(), du.clone(), layer.dw13.clone(), layer.dw2.clone(), layer.dcentroids.clone()]
        assert m.device_status() == 0
    for a, b in zip(res[m.MOE_DISPATCH_GATHER], res[m.MOE_DISPATCH_SCATTER]):
        assert torch.equal(_bits(a), _bits(b))
