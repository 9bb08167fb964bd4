"""The figures the pages print (tests/golden/deepseek_v3_pages.txt, each with
its place on the pages) against the configuration, the oracle and the
accumulation diagnostic."""
import os

import numpy as np
import torch

import oracle
import synthetic as S

HERE = os.path.dirname(os.path.abspath(__file__))


def _facts():
    out = {}
    for ln in open(os.path.join(HERE, "golden", "deepseek_v3_pages.txt")):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            k, v = (x.strip() for x in ln.split("="))
            out[k] = float(v) if "." in v else int(v)
    return out


def test_layer_shape_is_the_pages():
    f = _facts()
    for sh in (S.LAYER_V3, S.ROUTE_V3, *S.DECODE_V3):
        assert sh.N == f["routed_experts"] and sh.K == f["experts_per_token"]
    assert f["shared_experts"] == 1          # group N of the grouped GEMMs is the single shared expert
    # the group-limited decode routing keeps at most as many groups as the pages' node limit
    assert all(sh.topk_groups <= f["max_nodes_per_token"] for sh in S.DECODE_V3)


def test_oracle_scale_granularity_is_the_pages():
    f = _facts()
    x = S.normal((3, 512), 1.0, S.key(0, "golden-q"))
    q, s = oracle.quant_1x128(x)
    assert s.shape == (3 // f["activation_tile_rows"], 512 // f["activation_tile_cols"])
    w = S.normal((256, 384), 0.05, S.key(0, "golden-w"))
    q, s = oracle.quant_128x128(w)
    assert s.shape == (256 // f["weight_block_rows"], 384 // f["weight_block_cols"])
    # changing one value changes exactly one scale: the one of its tile / block
    x2 = x.clone()
    x2[1, 300] = 1000.0
    _, s2 = oracle.quant_1x128(x2)
    s1 = oracle.quant_1x128(x)[1]
    tile = 300 // f["activation_tile_cols"]
    assert (s2 != s1).sum() == 1 and s2[1, tile] != s1[1, tile]


def test_limited_accumulation_matches_the_printed_order():
    """An accumulator that keeps the printed number of bits over the printed
    inner dimension errs by up to the printed order of magnitude; promoting
    every printed interval in fp32 removes it."""
    f = _facts()
    K, bits, iv = f["limited_accumulation_inner_dim"], f["limited_accumulation_bits"], f["promotion_interval"]
    rng = np.random.Generator(np.random.PCG64(0))
    prod = np.abs(rng.standard_normal((64, K))) * np.abs(rng.standard_normal(K))[None, :] * 0.02
    exact = prod.sum(1)

    def trunc(x):
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(m * 2.0 ** bits) / 2.0 ** bits, e)

    acc = np.zeros(64)
    for k in range(K):
        acc = trunc(acc + prod[:, k])
    err = np.max(np.abs(acc - exact) / exact)
    assert f["limited_accumulation_max_rel_error"] / 10 < err < f["limited_accumulation_max_rel_error"] * 10
    part_sums = prod.reshape(64, K // iv, iv).astype(np.float32).sum(2, dtype=np.float32)
    promoted = part_sums.sum(1, dtype=np.float32)
    assert np.max(np.abs(promoted - exact) / exact) < 1e-5
