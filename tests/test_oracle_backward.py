"""Pins of the oracle's backward pass and training step (CPU only).

The backward's readings (oracle/moe_oracle.c, [train]): the gradient of the
layer formula h'_t = u_t + FFN_shared(u_t) + sum_k g_{t,k} FFN_{idx}(u_t)
(nlp-lineage.vercel.app "DeepSeek-V3 Technical Report (2024)", "The
notation") with the expert choice held fixed; the FP8 path quantises the
operands of every backward product with the tile rule of the learn.ifs.name
FP8 paragraph, along that product's own contraction dimension.

The pins do not restate the oracle's chain rule:
  * the FP64 mode (fp8=False) against central finite differences of an
    independent FP64 forward written below, in random directions of every
    parameter (u, centroids, each expert's W1, W3, W2);
  * the FP8 mode against the FP64 mode, on weights and tokens whose 128-blocks
    span a factor of 2^6 in magnitude, so that a scale taken from the wrong
    block or a transposed scale grid shows as an O(1) error, while correct
    FP8 rounding stays within a few per cent;
  * the new quantisers and the weight-gradient product against brute force
    (torch's float8_e4m3fn conversion, dequantise-then-multiply);
  * one training step as a descent step of the exact loss.
"""
import numpy as np
import pytest
import torch

import oracle

TINY = dict(T=7, d=256, N=4, K=2, I=256)


def _setup(T, d, N, K, I, seed=0, spread=False):
    """Seeded tiny layer: u, G bf16; centroids, weights fp32 (bf16-valued)."""
    rng = np.random.default_rng(seed)

    def bf(x):
        return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)

    def blocks(shape, std):
        w = rng.standard_normal(shape) * std
        if spread:   # every 128x128 block (or 128-column tile) its own magnitude, 2^-3 .. 2^3
            r, c = shape
            f = np.exp2(rng.integers(-3, 4, size=((r + 127) // 128, c // 128)))
            w *= np.repeat(np.repeat(f, 128, axis=0)[:r], 128, axis=1)
        return bf(w).float().numpy()

    u = bf(blocks((T, d), 1.0))
    G = bf(blocks((T, d), 0.5))
    E = (rng.standard_normal((N, d)) / np.sqrt(d)).astype(np.float32)
    W = [(blocks((I, d), 1 / np.sqrt(d)), blocks((I, d), 1 / np.sqrt(d)), blocks((d, I), 1 / np.sqrt(I)))
         for _ in range(N + 1)]
    bias = (rng.uniform(-0.01, 0.01, N)).astype(np.float32)
    return u, G, E, W, bias


def forward_exact(uv, E, W, idx, Gv):
    """L = sum(G * h') in FP64 with the expert choice idx held fixed: the
    layer formula written out token by token (independent of the oracle)."""
    T, d = uv.shape
    N = E.shape[0]

    def ffn(w, x):
        w1, w3, w2 = w
        h1, h3 = x @ w1.T, x @ w3.T
        return (h1 / (1.0 + np.exp(-h1)) * h3) @ w2.T

    L = 0.0
    for t in range(T):
        s = 1.0 / (1.0 + np.exp(-(E @ uv[t])))
        sel = idx[t]
        g = s[sel] / s[sel].sum()
        h = uv[t] + ffn(W[N], uv[t])
        for k, e in enumerate(sel):
            h = h + g[k] * ffn(W[e], uv[t])
        L += float(Gv[t] @ h)
    return L


def _exact_backward(u, G, E, W, bias, K):
    return oracle.layer_backward(u, E, bias, K, lambda e: W[e], G, fp8=False)


def test_backward_fp64_matches_finite_differences():
    T, d, N, K, I = TINY.values()
    u, G, E, W, bias = _setup(T, d, N, K, I, seed=1)
    bw = _exact_backward(u, G, E, W, bias, K)
    idx = bw.route.topk_idx
    uv = u.double().numpy()
    Gv = G.double().numpy()
    Wd = [tuple(w.astype(np.float64) for w in ws) for ws in W]
    Ed = E.astype(np.float64)
    rng = np.random.default_rng(7)
    eps = 1e-5

    def fd(f, x):
        v = rng.standard_normal(x.shape)
        return (f(x + eps * v) - f(x - eps * v)) / (2 * eps), v

    checks = []
    d_u, v = fd(lambda x: forward_exact(x, Ed, Wd, idx, Gv), uv)
    checks.append(("u", d_u, float((bw.du * v).sum())))
    d_e, v = fd(lambda x: forward_exact(uv, x, Wd, idx, Gv), Ed)
    checks.append(("centroids", d_e, float((bw.de * v).sum())))
    for e in range(N + 1):
        for j, (name, grad) in enumerate((("w1", bw.dw1[e]), ("w3", bw.dw3[e]), ("w2", bw.dw2[e]))):
            def f(x, e=e, j=j):
                Wx = list(Wd)
                ws = list(Wx[e])
                ws[j] = x
                Wx[e] = tuple(ws)
                return forward_exact(uv, Ed, Wx, idx, Gv)
            dd, v = fd(f, Wd[e][j])
            checks.append((f"{name}[{e}]", dd, float((grad * v).sum())))
    for name, num, ana in checks:
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (name, num, ana)


def test_backward_fp64_residual_and_zero_experts():
    """With every W2 zero the experts output nothing: du = G + the gate path
    (which vanishes too, since dg = G . y = 0), and dW1 = dW3 = 0."""
    T, d, N, K, I = TINY.values()
    u, G, E, W, bias = _setup(T, d, N, K, I, seed=2)
    W0 = [(w1, w3, np.zeros_like(w2)) for (w1, w3, w2) in W]
    for fp8 in (False, True):
        bw = oracle.layer_backward(u, E, bias, K, lambda e: W0[e], G, fp8=fp8)
        np.testing.assert_array_equal(bw.du, G.double().numpy())
        assert not bw.dw1.any() and not bw.dw3.any() and not bw.de.any() and not bw.dg.any()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def test_backward_fp8_close_to_fp64_with_spread_block_scales():
    """E4M3 keeps 3 mantissa bits: rounding moves an element by up to 2^-4 of
    itself (about 3.6 % rms), so a product of two quantised operands is off by
    about 5 % in norm, and the chain dY -> dA -> dH -> dX, dW compounds that to
    6-12 % here (measured: 4-7 % without the block spread, up to 12 % with
    it). A scale taken from the wrong block or a transposed scale grid
    (block magnitudes here differ by up to 2^6) gives errors of order one,
    and so does a wrong operand or sign; the bound is 0.2."""
    T, d, N, K, I = 300, 256, 4, 2, 256      # experts of ~150 rows: several 128-row blocks each
    u, G, E, W, bias = _setup(T, d, N, K, I, seed=3, spread=True)
    ex = _exact_backward(u, G, E, W, bias, K)
    q = oracle.layer_backward(u, E, bias, K, lambda e: W[e], G, fp8=True)
    np.testing.assert_array_equal(q.route.topk_idx, ex.route.topk_idx)
    errs = {"h": _rel(q.h, ex.h), "du": _rel(q.du, ex.du), "de": _rel(q.de, ex.de)}
    for e in range(N + 1):
        if ex.rows[e].size:
            errs[f"dw1[{e}]"] = _rel(q.dw1[e], ex.dw1[e])
            errs[f"dw3[{e}]"] = _rel(q.dw3[e], ex.dw3[e])
            errs[f"dw2[{e}]"] = _rel(q.dw2[e], ex.dw2[e])
    bad = {k: v for k, v in errs.items() if not v < 0.2}
    assert not bad, bad
    assert max(errs.values()) > 1e-4   # the FP8 path really quantised something


def test_quant_128x1_is_the_1x128_rule_on_the_transpose():
    rng = np.random.default_rng(4)
    for R, C in ((1, 128), (130, 256), (256, 128), (300, 384)):
        x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-6, 7, size=(R, C)))).astype(np.float32)
        x[:, 5] = 0.0
        q, s = oracle.quant_128x1(x)
        Rp = (R + 127) // 128 * 128
        xp = np.zeros((Rp, C), np.float32)
        xp[:R] = x
        q2, s2 = oracle.quant_1x128_f32(np.ascontiguousarray(xp.T))
        np.testing.assert_array_equal(q, q2)
        np.testing.assert_array_equal(s, s2.T)


def test_quant_128x128_f32_brute_force():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((200, 256)) * np.exp2(rng.integers(-4, 5, size=(200, 256)))).astype(np.float32)
    w[128:, 128:] = 0.0
    q, s = oracle.quant_128x128_f32(w)
    for br in range(2):
        for bc in range(2):
            blk = w[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            sc = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
            assert s[br, bc] == sc
            ref = torch.from_numpy((blk / sc).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(q[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128], ref)
    # on bf16 values it is the bf16 quantiser exactly
    wb = torch.from_numpy(w).to(torch.bfloat16)
    q1, s1 = oracle.quant_128x128(wb)
    q2, s2 = oracle.quant_128x128_f32(wb.float().numpy())
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)


def test_fp8_gemm_kscaled_is_dequantised_product():
    rng = np.random.default_rng(6)
    M, Nd, Kp = 64, 96, 384
    qa = rng.integers(0, 256, (M, Kp), dtype=np.uint8)
    qb = rng.integers(0, 256, (Nd, Kp), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 1      # no NaN codes
    qb[(qb & 0x7F) == 0x7F] = 2
    sa = rng.uniform(0.1, 4.0, (Kp // 128, M)).astype(np.float32)
    sb = rng.uniform(0.1, 4.0, (Kp // 128, Nd)).astype(np.float32)
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    A = vals[qa] * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    B = vals[qb] * np.repeat(sb.T.astype(np.float64), 128, axis=1)
    np.testing.assert_allclose(oracle.fp8_gemm_kscaled(qa, sa, qb, sb), A @ B.T, rtol=1e-12,
                               atol=1e-12 * np.abs(A).max() * np.abs(B).max() * Kp)


def test_swiglu_backward_finite_differences():
    rng = np.random.default_rng(8)
    h1, h3, da = rng.standard_normal((3, 50)) * 3
    d1, d3 = oracle.swiglu_backward(h1, h3, da)
    eps = 1e-6
    f = lambda a, b: a / (1 + np.exp(-a)) * b
    np.testing.assert_allclose(d1, da * (f(h1 + eps, h3) - f(h1 - eps, h3)) / (2 * eps), rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(d3, da * (f(h1, h3 + eps) - f(h1, h3 - eps)) / (2 * eps), rtol=1e-7, atol=1e-9)


def test_train_step_is_a_descent_step_of_the_exact_loss():
    T, d, N, K, I = TINY.values()
    u, G, E, W, bias = _setup(T, d, N, K, I, seed=9)
    masters = {"w1": np.stack([w[0] for w in W]), "w3": np.stack([w[1] for w in W]),
               "w2": np.stack([w[2] for w in W]), "e": E}
    lr = 1e-3
    new, new_bias, bw = oracle.train_step(u, masters, bias, K, G, lr, gamma=1e-3)
    idx = bw.route.topk_idx
    uv, Gv = u.double().numpy(), G.double().numpy()

    def loss(m):
        Wm = [(m["w1"][e].astype(np.float64), m["w3"][e].astype(np.float64), m["w2"][e].astype(np.float64))
              for e in range(N + 1)]
        return forward_exact(uv, m["e"].astype(np.float64), Wm, idx, Gv)

    L0, L1 = loss(masters), loss(new)
    # first-order decrease: lr * |grad|^2 (exact gradient), FP8 gradients within 10 %
    ex = _exact_backward(u, G, E, W, bias, K)
    g2 = sum(float((x ** 2).sum()) for x in (ex.dw1, ex.dw3, ex.dw2, ex.de))
    assert L1 < L0
    assert 0.8 * lr * g2 < L0 - L1 < 1.2 * lr * g2
    np.testing.assert_array_equal(new_bias, oracle.bias_update(bias, bw.route.loads, T, K, 1e-3))
    for k in masters:
        assert new[k].dtype == np.float32 and new[k].shape == masters[k].shape
