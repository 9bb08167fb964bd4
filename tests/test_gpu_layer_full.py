"""Full V3-shape layers on the GPU, checked on sampled tokens by the oracle.

  * the FP8 layer: T=8192, d=7168, 256 routed + 1 shared experts, I=2048,
    top-8, Zipf-skewed expert popularity; the oracle checks h' of 256 tokens
    (the first and last tokens routed to the hottest and to the coldest used
    expert, whose last rows sit in ragged tail tiles, plus seeded uniform
    tokens) and the routing, loads and bias update of all tokens;
  * the decode shapes T=64 and T=256 with group-limited routing (8 groups of
    32, top-4 groups by the sum of each group's two best biased affinities).
"""
import numpy as np
import pytest
import torch

import synthetic as S
from test_gpu_layer import _run_and_check

pytestmark = pytest.mark.gpu


def _sample(T, n, seed=5):
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.sort(rng.choice(T, n, replace=False))


def pick_256(idx, loads, n=256, seed=5):
    """256 tokens to check: the first and last token routed to the hottest expert
    and to the coldest expert with any load (the last rows of those groups sit in
    their last, ragged, 128-row tile; the coldest group is one ragged tile), then
    seeded uniform tokens up to n."""
    T = idx.shape[0]
    hot = int(np.argmax(loads))
    used = np.nonzero(loads)[0]
    cold = int(used[np.argmin(loads[used])])
    forced = []
    for e in (hot, cold):
        rows = np.nonzero((idx == e).any(axis=1))[0]
        forced += [int(rows[0]), int(rows[-1])]
    rng = np.random.Generator(np.random.PCG64(seed))
    rest = [t for t in rng.permutation(T) if t not in forced][: n - len(set(forced))]
    toks = np.unique(np.concatenate([forced, rest]).astype(np.int64))
    assert toks.size == n
    print(f"V3 layer: hottest expert {hot} ({loads[hot]} rows, {loads[hot] % 128} in its last tile), coldest used "
          f"expert {cold} ({loads[cold]} rows); checked tokens include {sorted(set(forced))}")
    return toks


def test_layer_v3_fp8_sampled_tokens():
    sh = S.LAYER_V3
    tau, n_diff = _run_and_check(sh, zipf=True, pick=pick_256)
    print(f"V3 layer: achieved tau {tau:.3e}, {n_diff} near-tie tokens routed differently")


@pytest.mark.parametrize("which", [0, 1])
def test_layer_v3_decode_group_limited(which):
    sh = S.DECODE_V3[which]
    tau, n_diff = _run_and_check(sh, zipf=True, u_seed=3)
    print(f"{sh.name}: achieved tau {tau:.3e}")


def test_layer_v3_gather_and_scatter_dispatch_agree():
    """At the V3 shape (Zipf-skewed groups, ragged tails), GEMM 1 gathering the
    quantised tokens and the permutation writing the grouped rows give the same
    h' bits."""
    import mixture_experts_layer_90_b300 as m
    from test_gpu_layer import _build
    sh = S.LAYER_V3
    layer = _build(sh, zipf=True)
    u = S.tokens(sh, seed=1).cuda()
    outs = {}
    for mode in (m.MOE_DISPATCH_GATHER, m.MOE_DISPATCH_SCATTER):
        layer._desc.dispatch = mode
        outs[mode] = layer.forward(u, update_bias=False).clone()
        assert m.device_status() == 0
    assert torch.equal(outs[m.MOE_DISPATCH_GATHER].view(torch.int16), outs[m.MOE_DISPATCH_SCATTER].view(torch.int16))
    del layer
    torch.cuda.empty_cache()
