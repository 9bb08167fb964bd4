"""Pins for the oracle's GEMMs, SwiGLU activation and combine.

The block-scaled GEMM follows the DeepSeek-V3 Technical Report summary
(learn.ifs.name), paragraphs on FP8 tiles and on FP32 promotion every 128
elements; the combine follows the layer formula in nlp-lineage.vercel.app,
"The notation".
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S


def _dec(codes: np.ndarray) -> np.ndarray:
    """E4M3 decode by torch (independent of the oracle's table)."""
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _rand_fp8(shape, name):
    v = S.normal(shape, 100.0, S.key(0, name, *shape), dtype=torch.float32).clamp(-448, 448)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _rand_scales(shape, name):
    return S.uniform(shape, 1e-4, 2e-2, S.key(0, name, *shape)).numpy()


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 130, 256), (128, 128, 512), (130, 256, 384)])
def test_fp8_gemm_brute_force(M, N, K):
    qa, qb = _rand_fp8((M, K), "a"), _rand_fp8((N, K), "b")
    sa = _rand_scales((M, K // 128), "sa")
    sb = _rand_scales(((N + 127) // 128, K // 128), "sb")
    C = oracle.fp8_gemm(qa, sa, qb, sb)
    A = _dec(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    B = _dec(qb) * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    ref = A @ B.T
    np.testing.assert_allclose(C, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_fp8_gemm_single_block_and_power_of_two_scaling():
    qa, qb = _rand_fp8((4, 128), "a1"), _rand_fp8((128, 128), "b1")
    sa = np.array([[0.5], [0.25], [3.0], [1e-3]], np.float32)
    sb = np.array([[0.125]], np.float32)
    C = oracle.fp8_gemm(qa, sa, qb, sb)
    exact = (_dec(qa) @ _dec(qb).T)          # integer-valued multiples of 2^-18: exact
    np.testing.assert_array_equal(C, exact * (sa.astype(np.float64) * 0.125))
    # a row scale times 2^k scales the output row by exactly 2^k
    sa2 = sa.copy()
    sa2[2, 0] *= 8.0
    C2 = oracle.fp8_gemm(qa, sa2, qb, sb)
    np.testing.assert_array_equal(C2[2], C[2] * 8.0)
    np.testing.assert_array_equal(C2[[0, 1, 3]], C[[0, 1, 3]])


def test_fp8_gemm_identity_weight_returns_dequantised_rows():
    qa = _rand_fp8((3, 256), "a2")
    sa = _rand_scales((3, 2), "sa2")
    one = np.uint8(0x38)                     # E4M3 code of 1.0
    qb = np.zeros((256, 256), np.uint8)
    qb[np.arange(256), np.arange(256)] = one
    sb = np.ones((2, 2), np.float32)
    C = oracle.fp8_gemm(qa, sa, qb, sb)
    np.testing.assert_array_equal(C, _dec(qa) * np.repeat(sa.astype(np.float64), 128, axis=1))


def test_bf16_gemm_brute_force():
    a = S.normal((7, 96), 1.0, S.key(0, "ga"))
    b = S.normal((33, 96), 0.1, S.key(0, "gb"))
    C = oracle.bf16_gemm(a, b)
    ref = a.double().numpy() @ b.double().numpy().T
    np.testing.assert_allclose(C, ref, rtol=1e-13, atol=1e-14)


def test_swiglu_identities():
    x = np.linspace(-30, 30, 601)
    one = np.ones_like(x)
    a = oracle.swiglu(x, one)
    # silu(x) - silu(-x) = x ; silu(0) = 0 ; silu -> x and -> 0 at the tails
    np.testing.assert_allclose(a - oracle.swiglu(-x, one), x, rtol=1e-14, atol=1e-14)
    assert oracle.swiglu(np.zeros(1), np.ones(1))[0] == 0.0
    assert abs(a[-1] - 30.0) < 1e-11 and abs(a[0]) < 1e-11
    # silu'(0) = 1/2: (silu(h) - silu(-h)) / 2h -> ... and silu(h)+silu(-h) = h*tanh(h/2)
    h = np.array([1e-3, 0.5, 2.0])
    np.testing.assert_allclose(oracle.swiglu(h, np.ones(3)) + oracle.swiglu(-h, np.ones(3)),
                               h * np.tanh(h / 2), rtol=1e-12)
    # the gate multiplies: h3 = 0 gives 0, h3 = 2 doubles
    np.testing.assert_array_equal(oracle.swiglu(x, np.zeros_like(x)), np.zeros_like(x))
    np.testing.assert_array_equal(oracle.swiglu(x, 2 * one), 2 * a)


def test_swiglu_quant_zero_and_tile_rule():
    R, I = 3, 256
    h1 = S.normal((R, I), 2.0, S.key(0, "h1"), dtype=torch.float32).double().numpy()
    h3 = S.normal((R, I), 2.0, S.key(0, "h3"), dtype=torch.float32).double().numpy()
    h3[1, :128] = 0.0
    q, s, dist, v = oracle.swiglu_quant(h1, h3)
    # a zero tile: scale 1 and every value +-0 (the sign of silu(h1) * 0 is kept)
    assert s[1, 0] == 1.0 and np.all((q[1, :128] & 0x7F) == 0)
    a32 = oracle.swiglu(h1, h3).astype(np.float32)
    q2, s2 = oracle.quant_1x128_f32(a32)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)
    assert np.all(dist >= 0)


def test_combine_closed_forms():
    T, d, K, R = 6, 64, 3, 40
    u = S.normal((T, d), 1.0, S.key(0, "cu"))
    ys = S.normal((T, d), 0.5, S.key(0, "cys"))
    y = S.normal((R, d), 0.5, S.key(0, "cy"))
    rng = np.random.Generator(np.random.PCG64(1))
    dest = np.stack([rng.choice(R, K, replace=False) for _ in range(T)]).astype(np.int32)
    g = rng.uniform(0.1, 1.0, (T, K))
    g /= g.sum(1, keepdims=True)
    out = oracle.combine(u, ys, y, g, dest)
    uf, ysf, yf = u.double().numpy(), ys.double().numpy(), y.double().numpy()
    ref = uf + ysf + np.einsum("tk,tkd->td", g, yf[dest])
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)
    # all expert outputs zero: h' == u exactly
    z = torch.zeros_like(y)
    np.testing.assert_array_equal(oracle.combine(u, torch.zeros_like(ys), z, g, dest), uf)
    # K = 1, g = 1: plain sum
    out1 = oracle.combine(u, ys, y, np.ones((T, 1)), dest[:, :1])
    np.testing.assert_allclose(out1, uf + ysf + yf[dest[:, 0]], rtol=1e-15)


def test_expert_ffn_fp8_matches_dequantised_float64_chain():
    d, I, R = 256, 128, 5
    x = S.normal((R, d), 1.0, S.key(0, "fx"))
    w1 = S.normal((I, d), d ** -0.5, S.key(0, "fw1"))
    w3 = S.normal((I, d), d ** -0.5, S.key(0, "fw3"))
    w2 = S.normal((d, I), I ** -0.5, S.key(0, "fw2"))
    xq, xs = oracle.quant_1x128(x)
    y, det = oracle.expert_ffn_fp8(xq, xs, w1, w3, w2, want_detail=True)
    # independent chain: torch decode, float64 matmul, the oracle's own codes for a
    X = _dec(xq) * np.repeat(xs.astype(np.float64), 128, 1)

    def deq_w(w):
        q, s = oracle.quant_128x128(w)
        return _dec(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0)[:w.shape[0]], 128, 1)

    h1, h3 = X @ deq_w(w1).T, X @ deq_w(w3).T
    a = h1 / (1 + np.exp(-h1)) * h3
    A = _dec(det["aq"]) * np.repeat(det["as_"].astype(np.float64), 128, 1)
    assert np.max(np.abs(A - a)) <= 2 ** -4 * np.max(np.abs(a)) * 1.01
    np.testing.assert_allclose(y, A @ deq_w(w2).T, rtol=1e-12, atol=1e-12)


def test_limited_accumulation_diagnostic():
    """The pages report ~14-bit tensor-core accumulation giving up to ~2%
    relative error at inner dimension 4096, removed by promoting partial sums
    to FP32 every 128 elements. Emulating an accumulator that keeps 14
    significant bits (truncating, a reading) shows errors of a few percent,
    while per-128 promotion in fp32 is orders of magnitude better: the 2e-3
    tolerance used for the GPU sits between the two."""
    rng = np.random.Generator(np.random.PCG64(0))
    K = 4096
    a = rng.standard_normal((64, K))
    b = np.abs(rng.standard_normal(K)) * 0.02        # same-sign terms make alignment loss visible
    a = np.abs(a)
    prod = a * b[None, :]
    exact = prod.sum(1)

    def trunc(x, bits):
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(m * 2.0 ** bits) / 2.0 ** bits, e)

    acc = np.zeros(64)
    for k in range(K):
        acc = trunc(acc + prod[:, k], 14)
    err14 = np.max(np.abs(acc - exact) / np.abs(exact))
    acc32 = np.zeros(64, np.float32)
    for kb in range(K // 128):
        part = np.zeros(64, np.float32)
        for k in range(kb * 128, kb * 128 + 128):
            part = (part + prod[:, k].astype(np.float32)).astype(np.float32)
        acc32 = (acc32 + part).astype(np.float32)
    err32 = np.max(np.abs(acc32 - exact) / np.abs(exact))
    assert 2e-3 < err14 < 0.2
    assert err32 < 1e-5


def _bruteforce_layer(u, cent, bias, K, weights):
    """The layer formula (nlp-lineage page, "The notation") on tiny inputs,
    written independently of the oracle: numpy FP64 routing, torch's
    float8_e4m3fn conversion for every 1x128 / 128x128 quantisation, FP64
    matmuls, bf16 rounding of each expert output by torch."""
    uf = u.double().numpy()
    z = uf @ cent.double().numpy().T
    s = 1.0 / (1.0 + np.exp(-z))
    key = s + bias.double().numpy()[None, :]
    T, d = uf.shape

    def q1x128(x32):                       # rows of fp32 values
        x = torch.as_tensor(x32, dtype=torch.float32).reshape(x32.shape[0], -1, 128)
        amax = x.abs().amax(-1, keepdim=True)
        sc = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
        q = (x / sc).to(torch.float8_e4m3fn).to(torch.float64)
        return (q * sc.double()).reshape(x32.shape[0], -1).numpy()

    def q128x128(w):
        x = w.float()
        r, c = x.shape
        xb = x.reshape(r // 128, 128, c // 128, 128)
        amax = xb.abs().amax(dim=(1, 3), keepdim=True)
        sc = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
        q = (xb / sc).to(torch.float8_e4m3fn).to(torch.float64)
        return (q * sc.double()).reshape(r, c).numpy()

    def ffn(xdq, e):
        w1, w3, w2 = weights(e)
        h1, h3 = xdq @ q128x128(w1).T, xdq @ q128x128(w3).T
        a = h1 / (1 + np.exp(-h1)) * h3
        y = q1x128(a.astype(np.float32)) @ q128x128(w2).T
        return torch.as_tensor(y).to(torch.float32).to(torch.bfloat16).double().numpy()

    X = q1x128(u.float().numpy())
    out = uf + ffn(X, cent.shape[0])
    for t in range(T):
        chosen = np.sort(np.argsort(-key[t], kind="stable")[:K])
        g = s[t, chosen] / s[t, chosen].sum()
        for k, e in enumerate(chosen):
            out[t] += g[k] * ffn(X[t:t + 1], e)[0]
    return out


def test_layer_composition_matches_independent_bruteforce():
    """oracle.layer_tokens (routing, 1x128 / 128x128 quantisation, SwiGLU FFNs,
    re-quantised intermediate, bf16 expert outputs, shared expert, gate-weighted
    sum) against the brute force above; the bias range is wide so that a bias
    leaking into the gate, a dropped shared expert or a swapped gate/up
    projection all show up far above the rounding differences."""
    sh = S.LayerShape(T=6, d=256, N=8, K=3, I=128, name="bf")
    u = S.tokens(sh)
    cent = S.centroids(sh)
    bias = S.uniform((sh.N,), -0.5, 0.5, S.key(7, "bf-bias"))
    wts = {e: S.expert_weights(sh, e) for e in range(sh.N + 1)}
    got, r, _ = oracle.layer_tokens(u, cent, bias, sh.K, lambda e: wts[e], np.arange(sh.T), fp8=True)
    ref = _bruteforce_layer(u, cent, bias, sh.K, lambda e: wts[e])
    scale = np.abs(ref - u.double().numpy()).max()
    # Both sides compute the same roundings; they may differ only in FP64 summation
    # order (~1e-16) or, were an expert output to land on a bf16 rounding boundary,
    # by the brute force's fp32 step there (none does for these seeded inputs).
    # A bias leaking into the gates moves them by ~0.18 here.
    assert np.max(np.abs(got - ref)) <= 1e-9 * scale, np.max(np.abs(got - ref)) / scale


def test_layer_with_zero_down_projections_returns_u():
    """W2 = 0 for every expert (routed and shared): h' equals u exactly."""
    sh = S.LayerShape(T=5, d=256, N=8, K=2, I=128, name="w2zero")
    u = S.tokens(sh)
    cent = S.centroids(sh)
    bias = S.bias(sh)

    def wts(e):
        w1, w3, w2 = S.expert_weights(sh, e)
        return w1, w3, torch.zeros_like(w2)
    for fp8 in (True, False):
        got, _, _ = oracle.layer_tokens(u, cent, bias, sh.K, wts, np.arange(sh.T), fp8=fp8)
        np.testing.assert_array_equal(got, u.double().numpy())


# --------------------------------------------------------------------------
# the bf16 expert path (the tiny layer and bf16_grouped_gemm's SwiGLU epilogue)
# --------------------------------------------------------------------------

def _bf16_rne(x: np.ndarray) -> np.ndarray:
    """Single rounding of FP64 values to bf16 (8 significant bits, ties to even),
    written from the definition: x = m * 2^e with 0.5 <= |m| < 1, so m * 2^8 is
    rounded to an integer by numpy's round-half-to-even. No subnormal or overflow
    case arises at these magnitudes."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.round(m * 256.0), e - 8)


def _bruteforce_bf16_ffn(x, w1, w3, w2, swap_gate_up=False, round_a=True):
    """SwiGLU expert W2 (silu(W1 x) * W3 x) on bf16 values, products exact in FP64;
    the intermediate a is rounded once to bf16 (where the bf16 kernels store it)."""
    xf, w1f, w3f, w2f = (t.double().numpy() for t in (x, w1, w3, w2))
    h1, h3 = xf @ w1f.T, xf @ w3f.T
    if swap_gate_up:
        h1, h3 = h3, h1
    a = h1 / (1.0 + np.exp(-h1)) * h3
    if round_a:
        a = _bf16_rne(a)
    return a @ w2f.T


def _bruteforce_bf16_layer(u, cent, bias, K, weights, **ffn_kw):
    """The layer formula (nlp-lineage page, "The notation") with bf16 experts,
    written independently of the oracle: numpy FP64 routing (sigmoid affinity,
    top-K of s + b by a stable sort, gates s / sum s over the chosen), each expert
    output rounded once to bf16, then u + shared + sum_k g_k y_k in FP64."""
    uf = u.double().numpy()
    s = 1.0 / (1.0 + np.exp(-(uf @ cent.double().numpy().T)))
    key = s + bias.double().numpy()[None, :]
    out = uf + _bf16_rne(_bruteforce_bf16_ffn(u, *weights(cent.shape[0]), **ffn_kw))
    for t in range(uf.shape[0]):
        chosen = np.sort(np.argsort(-key[t], kind="stable")[:K])
        g = s[t, chosen] / s[t, chosen].sum()
        for k, e in enumerate(chosen):
            out[t] += g[k] * _bf16_rne(_bruteforce_bf16_ffn(u[t:t + 1], *weights(e), **ffn_kw))[0]
    return out


def _bf16_case():
    sh = S.LayerShape(T=6, d=256, N=8, K=3, I=128, fp8=False, centroid_f32=False, name="bf16-bf")
    u = S.tokens(sh)
    cent = S.centroids(sh)
    bias = S.uniform((sh.N,), -0.5, 0.5, S.key(9, "bf16-bf-bias"))   # wide: a bias leaking into g shows
    wts = {e: S.expert_weights(sh, e) for e in range(sh.N + 1)}
    return sh, u, cent, bias, (lambda e: wts[e])


def test_bf16_rounding_helper_is_a_single_rne_rounding():
    """The brute force's own bf16 rounding against exactly representable cases:
    bf16 values are fixed points, midpoints go to the even neighbour, and any other
    value goes to the nearer neighbour."""
    bf = torch.tensor([1.0, 1.0078125, -3.5, 448.0, 2.0 ** -20], dtype=torch.float64)
    np.testing.assert_array_equal(_bf16_rne(bf.numpy()), bf.numpy())
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even mantissa (1)
    assert _bf16_rne(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    assert _bf16_rne(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    assert _bf16_rne(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1.0 + 2.0 ** -7
    # agrees with the oracle's C rounding on values away from fp32 double-rounding cases
    x = S.normal((4096,), 3.0, S.key(0, "bf16-rne"), dtype=torch.float32).double().numpy() * (1 + 2.0 ** -30)
    np.testing.assert_array_equal(_bf16_rne(x), oracle.bf16_value(oracle.bf16_round(x)))


def test_expert_ffn_bf16_matches_independent_bruteforce():
    """oracle.expert_ffn_bf16 (FP64 products, a rounded to bf16, y unrounded)
    against the brute force; a swapped gate/up projection or a missing rounding
    of a moves the result far beyond the agreement of the two."""
    sh, u, cent, bias, wts = _bf16_case()
    w1, w3, w2 = wts(2)
    got = oracle.expert_ffn_bf16(u, w1, w3, w2)
    ref = _bruteforce_bf16_ffn(u, w1, w3, w2)
    scale = np.abs(ref).max()
    assert np.max(np.abs(got - ref)) <= 1e-12 * scale
    swapped = _bruteforce_bf16_ffn(u, w1, w3, w2, swap_gate_up=True)
    unrounded = _bruteforce_bf16_ffn(u, w1, w3, w2, round_a=False)
    assert np.max(np.abs(swapped - ref)) > 1e-2 * scale
    assert np.max(np.abs(unrounded - ref)) > 1e-5 * scale


def test_layer_bf16_composition_matches_independent_bruteforce():
    """oracle.layer_tokens(fp8=False): routing, bf16 SwiGLU experts with a and y
    rounded to bf16, the shared expert with gate 1, the gate-weighted sum, against
    the brute force above. The wide bias range makes a bias leaking into the gates,
    a dropped shared expert or a swapped gate/up projection show far above the
    FP64 summation-order differences the two may have."""
    sh, u, cent, bias, wts = _bf16_case()
    got, r, _ = oracle.layer_tokens(u, cent, bias, sh.K, wts, np.arange(sh.T), fp8=False)
    ref = _bruteforce_bf16_layer(u, cent, bias, sh.K, wts)
    scale = np.abs(ref - u.double().numpy()).max()
    assert np.max(np.abs(got - ref)) <= 1e-12 * scale, np.max(np.abs(got - ref)) / scale
    swapped = _bruteforce_bf16_layer(u, cent, bias, sh.K, wts, swap_gate_up=True)
    assert np.max(np.abs(swapped - ref)) > 1e-2 * scale
    # the bias steers the choice here: some token's set differs from the unbiased top-K
    s = 1.0 / (1.0 + np.exp(-(u.double().numpy() @ cent.double().numpy().T)))
    unbiased = np.sort(np.argsort(-s, axis=1, kind="stable")[:, :sh.K], axis=1)
    assert np.any(unbiased != r.topk_idx)
