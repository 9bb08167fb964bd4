"""Pins for the oracle's sequence-wise balance statistics.

The learn.ifs.name summary of the DeepSeek-V3 Technical Report (bias
paragraph) says that beside the per-expert bias only a tiny sequence-wise
balancing loss remains, against extreme imbalance inside one sequence; the
pages give no formula. The reading used here: for a sequence of T_s tokens,
f_i = N * (pairs routed to i) / (K * T_s), P_i = the mean over the sequence of
s_i / sum_j s_j, statistic = sum_i f_i P_i (the loss weight is the caller's).
"""
import numpy as np
import pytest

import oracle
import synthetic as S


def _case(T, N, K, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.standard_normal((T, N))
    s = 1.0 / (1.0 + np.exp(-z))
    idx = np.sort(np.argsort(-s, axis=1, kind="stable")[:, :K], axis=1).astype(np.int32)
    return s, idx


def _bruteforce(s, idx, K, seq_len):
    T, N = s.shape
    out_l, out_p, out_s = [], [], []
    for t0 in range(0, T, seq_len):
        ss, ii = s[t0:t0 + seq_len], idx[t0:t0 + seq_len]
        Ts = ss.shape[0]
        loads = np.bincount(ii.ravel(), minlength=N)
        P = (ss / ss.sum(axis=1, keepdims=True)).mean(axis=0)
        f = N * loads / (K * Ts)
        out_l.append(loads)
        out_p.append(P)
        out_s.append(float(np.dot(f, P)))
    return np.array(out_l), np.array(out_p), np.array(out_s)


@pytest.mark.parametrize("T,N,K,seq_len", [(10, 8, 2, 4), (300, 64, 6, 128), (512, 256, 8, 512), (7, 5, 3, 100)])
def test_matches_bruteforce_with_ragged_last_sequence(T, N, K, seq_len):
    s, idx = _case(T, N, K, seed=T)
    loads, prob, stat = oracle.seq_balance(s, idx, K, seq_len)
    bl, bp, bs = _bruteforce(s, idx, K, seq_len)
    np.testing.assert_array_equal(loads, bl)
    np.testing.assert_allclose(prob, bp, rtol=1e-13, atol=0)
    np.testing.assert_allclose(stat, bs, rtol=1e-13, atol=0)


def test_invariants():
    """Per sequence: the loads sum to K*T_s, the P_i sum to 1, the f_i sum to N."""
    T, N, K, L = 1000, 64, 6, 96
    s, idx = _case(T, N, K, seed=1)
    loads, prob, stat = oracle.seq_balance(s, idx, K, L)
    lens = np.array([min(L, T - t0) for t0 in range(0, T, L)])
    np.testing.assert_array_equal(loads.sum(axis=1), K * lens)
    np.testing.assert_allclose(prob.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose((N * loads / (K * lens[:, None])).sum(axis=1), N, rtol=1e-12)


def test_uniform_affinities_give_one():
    """Equal affinities make every P_i = 1/N, so the statistic is sum f_i / N = 1
    whatever the routing."""
    T, N, K = 200, 32, 4
    s = np.full((T, N), 0.3)
    _, idx = _case(T, N, K, seed=2)
    _, prob, stat = oracle.seq_balance(s, idx, K, 64)
    np.testing.assert_allclose(prob, 1.0 / N, rtol=1e-14)
    np.testing.assert_allclose(stat, 1.0, rtol=1e-13)


def test_balanced_loads_give_one_and_collapse_gives_n_over_k():
    """Balanced loads (every f_i = 1) give sum P_i = 1; every token sending its K
    pairs to the same experts, with all affinity on them, gives the largest
    value, (N/K) * K * (1/K) = N/K."""
    N, K, T = 16, 4, 64
    # balanced: token t picks experts 4(t % 4) .. 4(t % 4) + 3, so every expert gets T*K/N pairs
    idx = np.array([[4 * (t % 4) + k for k in range(K)] for t in range(T)], np.int32)
    s, _ = _case(T, N, K, seed=3)
    loads, _, stat = oracle.seq_balance(s, idx, K, T)
    assert (loads == T * K // N).all()
    np.testing.assert_allclose(stat, 1.0, rtol=1e-13)
    # collapse: experts 0..K-1 for every token, affinity only there
    idx = np.tile(np.arange(K, dtype=np.int32), (T, 1))
    s = np.zeros((T, N))
    s[:, :K] = 0.7
    _, prob, stat = oracle.seq_balance(s, idx, K, T)
    np.testing.assert_allclose(prob[0, :K], 1.0 / K, rtol=1e-14)
    np.testing.assert_allclose(stat, N / K, rtol=1e-13)


def test_normalises_over_all_experts_not_the_chosen():
    """P_i divides by the sum over all N affinities: dividing by the chosen
    experts' sum (the gate normalisation) gives a different, larger value."""
    T, N, K = 50, 32, 4
    s, idx = _case(T, N, K, seed=4)
    _, prob, _ = oracle.seq_balance(s, idx, K, T)
    chosen_sum = np.take_along_axis(s, idx, axis=1).sum(axis=1, keepdims=True)
    wrong = (s / chosen_sum).mean(axis=0)
    assert np.max(np.abs(prob[0] - wrong)) > 0.1 * np.max(prob[0])
