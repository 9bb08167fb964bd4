"""Pins for the oracle's routing, permutation and bias update.

Facts from the pages (DeepSeek-V3 Technical Report summaries):
  * learn.ifs.name, MoE paragraph: top-K by sigmoid affinity to the expert's
    centroid, gates normalised over the chosen experts;
  * same page, bias paragraph: the bias enters the top-K choice only, the gate
    uses the raw score; after a step, overloaded experts' bias falls by gamma,
    underloaded ones' rises;
  * nlp-lineage.vercel.app, "The notation": chosen iff s + b is in the top 8;
  * same page, load-balancing item: no token is dropped.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S


def _tiny(T=24, d=64, N=16, seed=0, f32=True):
    u = S.normal((T, d), 1.0, S.key(seed, "ru", T, d))
    e = S.normal((N, d), 1.0 / np.sqrt(d), S.key(seed, "re", N, d),
                 dtype=torch.float32 if f32 else torch.bfloat16)
    b = S.uniform((N,), -0.01, 0.01, S.key(seed, "rb", N))
    return u, e, b


def _brute_topk(u, e, b, K, n_groups=1, topk_groups=1):
    uf = u.to(torch.float64).numpy()
    ef = e.to(torch.float64).numpy()
    z = uf @ ef.T
    s = 1.0 / (1.0 + np.exp(-z))
    key = s + b.to(torch.float64).numpy()[None, :]
    T, N = key.shape
    idx = np.empty((T, K), np.int64)
    for t in range(T):
        allowed = np.arange(N)
        if n_groups > 1:
            per = N // n_groups
            gs = []
            for g in range(n_groups):
                kk = np.sort(key[t, g * per:(g + 1) * per])[::-1]
                gs.append(kk[0] + kk[1])
            order = np.lexsort((np.arange(n_groups), -np.array(gs)))
            keep = np.sort(order[:topk_groups])
            allowed = np.concatenate([np.arange(g * per, (g + 1) * per) for g in keep])
        order = np.lexsort((allowed, -key[t, allowed]))
        idx[t] = np.sort(allowed[order[:K]])
    return idx, s


@pytest.mark.parametrize("f32", [True, False])
def test_route_matches_brute_force(f32):
    u, e, b = _tiny(f32=f32)
    r = oracle.route(u, e, b, K=4, want_scores=True)
    idx, s = _brute_topk(u, e, b, 4)
    np.testing.assert_array_equal(r.topk_idx, idx)
    np.testing.assert_allclose(r.scores, s, rtol=1e-13, atol=0)
    g_ref = np.take_along_axis(s, idx, 1)
    g_ref = g_ref / g_ref.sum(1, keepdims=True)
    np.testing.assert_allclose(r.gates, g_ref, rtol=1e-13)
    np.testing.assert_array_equal(r.loads, np.bincount(idx.ravel(), minlength=16))


def test_group_limited_matches_brute_force_and_reduces_to_flat():
    u, e, b = _tiny(T=40, d=64, N=32)
    r = oracle.route(u, e, b, K=4, n_groups=8, topk_groups=3)
    idx, _ = _brute_topk(u, e, b, 4, n_groups=8, topk_groups=3)
    np.testing.assert_array_equal(r.topk_idx, idx)
    flat = oracle.route(u, e, b, K=4)
    for ng in (1, 8):
        r2 = oracle.route(u, e, b, K=4, n_groups=ng, topk_groups=ng)
        np.testing.assert_array_equal(r2.topk_idx, flat.topk_idx)
        np.testing.assert_array_equal(r2.gates, flat.gates)
    # chosen experts all lie in at most topk_groups groups
    assert np.all(np.array([len(set(row // 4)) for row in r.topk_idx]) <= 3)


def test_gates_sum_to_one_and_k_distinct():
    u, e, b = _tiny(T=64)
    r = oracle.route(u, e, b, K=6)
    np.testing.assert_allclose(r.gates.sum(1), 1.0, rtol=0, atol=4e-16)
    assert np.all(r.gates > 0)
    assert all(len(set(row)) == 6 for row in r.topk_idx)
    assert np.all(np.diff(r.topk_idx, axis=1) > 0)
    assert r.loads.sum() == 64 * 6


def test_zero_bias_selects_top_logits():
    u, e, _ = _tiny(T=32)
    r = oracle.route(u, e, np.zeros(16, np.float32), K=4)
    z = u.to(torch.float64).numpy() @ e.to(torch.float64).numpy().T
    top = np.sort(np.argsort(-z, axis=1, kind="stable")[:, :4], axis=1)
    np.testing.assert_array_equal(r.topk_idx, top)


def test_bias_changes_choice_not_gate_value():
    u, e, b = _tiny(T=32)
    r0 = oracle.route(u, e, b, K=4)
    # a common shift of every bias keeps every choice, so gates stay bit-equal
    r1 = oracle.route(u, e, (b.double() + 0.25).float(), K=4)
    np.testing.assert_array_equal(r0.topk_idx, r1.topk_idx)
    np.testing.assert_array_equal(r0.gates, r1.gates)
    # force experts 3, 7, 9, 12 in: every token takes them, gates use raw s
    bf = b.clone()
    bf[[3, 7, 9, 12]] = 10.0
    r2 = oracle.route(u, e, bf, K=4, want_scores=True)
    assert np.all(r2.topk_idx == np.array([3, 7, 9, 12]))
    s = r2.scores[:, [3, 7, 9, 12]]
    np.testing.assert_allclose(r2.gates, s / s.sum(1, keepdims=True), rtol=1e-15)
    assert r2.loads[[3, 7, 9, 12]].tolist() == [32] * 4
    # push two experts out: load 0, every token still gets K experts (no drops)
    bn = b.clone()
    bn[[0, 5]] = -10.0
    r3 = oracle.route(u, e, bn, K=4)
    assert r3.loads[0] == 0 and r3.loads[5] == 0 and r3.loads.sum() == 32 * 4


def test_one_hot_token_logits_are_centroid_entries():
    d, N = 64, 16
    _, e, _ = _tiny(d=d, N=N)
    u = torch.zeros((1, d), dtype=torch.bfloat16)
    u[0, 5] = 1.0
    r = oracle.route(u, e, np.zeros(N, np.float32), K=2, want_scores=True)
    z = e[:, 5].double().numpy()
    np.testing.assert_allclose(r.scores[0], 1.0 / (1.0 + np.exp(-z)), rtol=1e-15)


def test_tie_goes_to_lower_index_and_near_tie_flag():
    d, N = 8, 8
    e = torch.zeros((N, d), dtype=torch.float32)
    u = torch.ones((1, d), dtype=torch.bfloat16)
    r = oracle.route(u, e, np.zeros(N, np.float32), K=3, delta=1e-9)
    assert r.topk_idx[0].tolist() == [0, 1, 2]       # all keys equal
    assert r.near_tie[0] and r.key_gap[0] == 0.0
    np.testing.assert_array_equal(r.gates[0], [1 / 3] * 3)


def test_k1_gate_is_exactly_one():
    u, e, b = _tiny()
    r = oracle.route(u, e, b, K=1)
    assert np.all(r.gates == 1.0)


def test_permute_invariants_and_stable_sort():
    rng = np.random.Generator(np.random.PCG64(5))
    T, N, K = 300, 12, 3
    idx = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(T)]).astype(np.int32)
    off, perm, dest = oracle.permute(idx, N)
    cnt = np.bincount(idx.ravel(), minlength=N)
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(cnt)]))
    # brute force: stable argsort of the flattened expert ids
    order = np.argsort(idx.ravel(), kind="stable")
    np.testing.assert_array_equal(perm, order // K)
    assert np.all(perm[dest] == np.arange(T)[:, None])
    for i in range(N):
        seg = perm[off[i]:off[i + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(idx[seg].__eq__(i).any(1))
    assert sorted(dest.ravel().tolist()) == list(range(T * K))


def test_permute_empty_experts():
    idx = np.array([[2, 5]] * 4, np.int32)
    off, perm, dest = oracle.permute(idx, 8)
    assert off.tolist() == [0, 0, 0, 4, 4, 4, 8, 8, 8]
    assert perm.tolist() == [0, 1, 2, 3, 0, 1, 2, 3]
    assert dest.tolist() == [[0, 4], [1, 5], [2, 6], [3, 7]]


def test_bias_update_closed_form():
    T, K, N = 10, 4, 8          # mean load 5
    loads = np.array([5, 6, 4, 0, 40, 5, 0, 0], np.int32)
    b = np.array([0.0, 0.01, -0.01, 0.5, -0.5, 1e-8, 3.0, -3.0], np.float32)
    g = np.float32(1e-3)
    out = oracle.bias_update(b, loads, T, K, 1e-3)
    exp = b.copy()
    for i, ld in enumerate(loads):
        if ld * N > T * K:
            exp[i] = np.float32(b[i] - g)
        elif ld * N < T * K:
            exp[i] = np.float32(b[i] + g)
    np.testing.assert_array_equal(out, exp)
    assert out[0] == b[0] and out[5] == b[5]          # at the mean: unchanged
    assert out[1] < b[1] and out[2] > b[2]


def test_bias_update_non_integer_mean():
    # T*K/N = 7.5: loads 7 -> raise, 8 -> lower
    out = oracle.bias_update(np.zeros(4, np.float32), np.array([7, 8, 7, 8], np.int32), T=10, K=3, gamma=0.5)
    np.testing.assert_array_equal(out, [0.5, -0.5, 0.5, -0.5])
