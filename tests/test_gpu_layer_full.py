"""Full V3-shape layers on the GPU, checked on sampled tokens by the oracle.

  * the FP8 layer: T=8192, d=7168, 256 routed + 1 shared experts, I=2048,
    top-8, Zipf-skewed expert popularity; the oracle checks 256 sampled tokens
    (seeded uniform, plus the first tokens routed to the hottest and to the
    coldest used expert) and the routing of all tokens;
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


def test_layer_v3_fp8_sampled_tokens():
    sh = S.LAYER_V3
    toks = _sample(sh.T, 254)
    tau, n_diff = _run_and_check(sh, tokens=toks, zipf=True)
    print(f"V3 layer: achieved tau {tau:.3e}, {n_diff} near-tie tokens routed differently")


@pytest.mark.parametrize("which", [0, 1])
def test_layer_v3_decode_group_limited(which):
    sh = S.DECODE_V3[which]
    tau, n_diff = _run_and_check(sh, zipf=True, u_seed=3)
    print(f"{sh.name}: achieved tau {tau:.3e}")
