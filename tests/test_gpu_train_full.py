"""The backward pass at the full V3 shape (T=8192, d=7168, 256 routed + 1
shared experts, top-8, I=2048, Zipf-skewed expert popularity), in the launch
configuration the benchmark times, checked against the oracle on what it can
compute from a sample.

  * Per token. The dgrad chain of a row (dY, dA, dH, dX) and the gate
    backward only involve that row's own values, so du_t, and a token's
    share of the centroid gradient, follow from the token alone. With
    dL/dh' = G zero except on three sampled tokens, the other tokens' du is
    exactly zero, every expert those tokens do not reach gets exactly zero
    weight gradients, and du of the sampled tokens and the centroid gradient
    match the oracle's backward of those three tokens.
  * Per expert. An expert's weight gradient involves all of its rows (its
    weight-gradient operands are scaled per 128 of its rows), and only them.
    With a full G, the coldest used expert's weight gradients match the
    oracle's backward of the tokens routed to it (weight gradients of that
    expert only), and so does du of those tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from test_gpu_train import TAU_BWD, _rowwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v3():
    import mixture_experts_layer_90_b300 as m
    sh = S.LAYER_V3
    cent = S.centroids(sh, zipf=True).cuda()
    bias = S.bias(sh).cuda()
    layer = m.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias, lambda e: S.expert_weights(sh, e, device="cuda"),
                             fp8=True, train=True, gamma=sh.gamma)
    u = S.tokens(sh, seed=7)
    idx = torch.empty((sh.T, sh.K), dtype=torch.int32, device="cuda")
    layer.forward_train(u.cuda(), topk_idx=idx, update_bias=False)
    assert m.device_status() == 0
    cache = {}

    def weights(e):
        if e not in cache:
            cache[e] = tuple(w.cpu() for w in S.expert_weights(sh, e, device="cuda"))
        return cache[e]
    yield sh, layer, u, idx.cpu().numpy(), weights
    del layer
    torch.cuda.empty_cache()


def _oracle(sh, layer, u, toks, G, weights, wgrad_experts):
    b0 = layer.bias.cpu().numpy()
    ut = u[torch.as_tensor(toks)]
    r = oracle.route(ut, layer.centroids.cpu(), b0, sh.K, want_scores=True)
    assert not r.near_tie.any()
    return r, oracle.layer_backward(ut, layer.centroids.cpu(), b0, sh.K, weights, G[torch.as_tensor(toks)], fp8=True,
                                    route_all=r, stack=False, wgrad_experts=wgrad_experts)


def test_backward_v3_sampled_tokens(v3):
    import mixture_experts_layer_90_b300 as m
    sh, layer, u, idx, weights = v3
    T, d, N, K, I = sh.T, sh.d, sh.N, sh.K, sh.I
    rng = np.random.Generator(np.random.PCG64(11))
    toks = np.sort(rng.choice(T, 3, replace=False))
    G = torch.zeros((T, d), dtype=torch.bfloat16)
    G[torch.as_tensor(toks)] = S.grad_out(S.LayerShape(T=3, d=d, N=N, K=K, I=I), seed=12)
    du = layer.backward(u.cuda(), G.cuda())
    assert m.device_status() == 0
    r, ref = _oracle(sh, layer, u, toks, G, weights, wgrad_experts=set())
    np.testing.assert_array_equal(r.topk_idx, idx[toks])
    du = du.cpu().float().numpy()
    assert not du[np.setdiff1d(np.arange(T), toks)].any(), "a token with a zero gradient row got a nonzero du"
    reached = sorted(set(r.topk_idx.ravel().tolist()))
    untouched = torch.ones(N + 1, dtype=torch.bool)
    untouched[torch.as_tensor(reached + [N])] = False
    assert not layer.dw13[untouched].any() and not layer.dw2[untouched].any()
    de = layer.dcentroids.cpu().numpy()
    assert not de[np.setdiff1d(np.arange(N), reached)].any()
    errs = {"du": _rowwise(du[toks], ref.du, "du"), "de": _rowwise(de[reached], ref.de[reached], "de")}
    print(f"V3 backward, tokens {toks.tolist()} reaching {len(reached)} experts: {errs}")
    assert max(errs.values()) < TAU_BWD, errs


def test_backward_v3_coldest_expert_weight_gradients(v3):
    import mixture_experts_layer_90_b300 as m
    sh, layer, u, idx, weights = v3
    T, d, N, K, I = sh.T, sh.d, sh.N, sh.K, sh.I
    G = S.grad_out(sh, seed=13)
    du = layer.backward(u.cuda(), G.cuda())
    assert m.device_status() == 0
    loads = np.bincount(idx.ravel(), minlength=N)
    used = np.nonzero(loads)[0]
    e = int(used[np.argmin(loads[used])])
    toks = np.nonzero((idx == e).any(axis=1))[0]
    r, ref = _oracle(sh, layer, u, toks, G, weights, wgrad_experts={e})
    np.testing.assert_array_equal(r.topk_idx, idx[toks])
    dw13 = layer.dw13[e].view(I // 128, 2, 128, d)
    errs = {"dw1": _rowwise(dw13[:, 0].reshape(I, d).cpu().numpy(), ref.dw1[e], "dw1"),
            "dw3": _rowwise(dw13[:, 1].reshape(I, d).cpu().numpy(), ref.dw3[e], "dw3"),
            "dw2": _rowwise(layer.dw2[e].cpu().numpy(), ref.dw2[e], "dw2"),
            "du": _rowwise(du[torch.as_tensor(toks).cuda()].cpu().float().numpy(), ref.du, "du")}
    print(f"V3 backward, coldest used expert {e} ({loads[e]} rows, {toks.size} tokens): {errs}")
    assert max(errs.values()) < TAU_BWD, errs
