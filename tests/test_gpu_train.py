"""The backward pass and the training step on the GPU against the oracle.

Readings (include/moe.h, "Training"; oracle/moe_oracle.c, [train]): the
gradient of the layer formula (nlp-lineage.vercel.app "DeepSeek-V3 Technical
Report (2024)", "The notation") with the expert choice held fixed, the
backward's products on FP8 operands scaled along their own contraction
(learn.ifs.name, FP8 paragraph), plain SGD on fp32 masters, and the bias
update after each step (learn.ifs.name, bias paragraph).

Bars: integer and byte work bit-exact (transposes, SGD and its 128x128
re-quantisation, K-block offsets, routing, loads, bias); products and
gradients normwise per row against the oracle's FP64 values, at tolerances
stated beside each check.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import check_bf16

pytestmark = pytest.mark.gpu


def _lib():
    import mixture_experts_layer_90_b300 as m
    return m


def _vals():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _codes(rng, shape):
    q = rng.integers(0, 256, shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38   # no NaN codes
    return q


def _rowwise(got, exp, what):
    """max over rows of |got - exp| / max|exp| of the row (0 for zero rows)."""
    got, exp = np.asarray(got, np.float64), np.asarray(exp, np.float64)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    g2, e2 = got.reshape(-1, got.shape[-1]), exp.reshape(-1, exp.shape[-1])
    m = np.abs(e2).max(axis=1)
    err = np.abs(g2 - e2).max(axis=1)
    zero = m == 0
    assert np.all(err[zero] == 0), f"{what}: nonzero where the oracle has zeros"
    return float(np.max(err[~zero] / m[~zero])) if (~zero).any() else 0.0


# --------------------------------------------------------------------------
# kernels
# --------------------------------------------------------------------------

def test_fp8_transpose_128x128_bit_exact():
    m = _lib()
    rng = np.random.default_rng(0)
    G, rows, cols = 3, 256, 384
    q = _codes(rng, (G, rows, cols))
    s = rng.uniform(0.01, 2.0, (G, rows // 128, cols // 128)).astype(np.float32)
    qt, st = m.fp8_transpose_128x128(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    np.testing.assert_array_equal(qt.cpu().numpy(), q.transpose(0, 2, 1))
    np.testing.assert_array_equal(st.cpu().numpy(), s.transpose(0, 2, 1))


def test_sgd_requant_bit_exact():
    """New master fl32(w - fl32(lr g)), its 128x128 quantisation and the
    transposed copy, all bit for bit against the oracle's."""
    m = _lib()
    rng = np.random.default_rng(1)
    G, rows, cols = 2, 256, 384
    w = (rng.standard_normal((G, rows, cols)) * np.exp2(rng.integers(-3, 4, (G, rows, cols)))).astype(np.float32)
    w[1, :128, :128] = 0.0
    g = (rng.standard_normal((G, rows, cols)) * 10).astype(np.float32)
    g[1, :128, :128] = 0.0   # an all-zero block: scale 1
    lr = 3e-3
    wd, gd = torch.from_numpy(w).cuda(), torch.from_numpy(g).cuda()
    q = torch.empty((G, rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty((G, rows // 128, cols // 128), dtype=torch.float32, device="cuda")
    qt = torch.empty((G, cols, rows), dtype=torch.uint8, device="cuda")
    st = torch.empty((G, cols // 128, rows // 128), dtype=torch.float32, device="cuda")
    m.moe_sgd_requant_128x128(wd, gd, lr, q, s, qt, st)
    w_new = oracle.sgd_f32(w, g, lr)
    np.testing.assert_array_equal(wd.cpu().numpy(), w_new)
    for e in range(G):
        qe, se = oracle.quant_128x128_f32(w_new[e])
        np.testing.assert_array_equal(q[e].cpu().numpy(), qe)
        np.testing.assert_array_equal(s[e].cpu().numpy(), se)
        np.testing.assert_array_equal(qt[e].cpu().numpy(), qe.T)
        np.testing.assert_array_equal(st[e].cpu().numpy(), se.T)
    assert s[1, 0, 0].item() == 1.0


def test_sgd_f32_bit_exact():
    m = _lib()
    rng = np.random.default_rng(2)
    w = rng.standard_normal(1000).astype(np.float32)
    g = rng.standard_normal(1000).astype(np.float32)
    wd = torch.from_numpy(w).cuda()
    m.moe_sgd_f32(wd, torch.from_numpy(g).cuda(), 0.37)
    np.testing.assert_array_equal(wd.cpu().numpy(), oracle.sgd_f32(w, g, 0.37))


@pytest.mark.parametrize("blocks", [[2, 0, 1, 3, 1], [0, 0, 1], [5]])
def test_wgrad_gemm_against_oracle(blocks):
    """Groups split K (empty groups included): fp32 out within 1e-5 of the
    row's largest value (products of E4M3 values are exact in fp32; the
    tensor cores sum 128 of them per block in fp32, the epilogue adds the
    scaled block sums in fp32)."""
    m = _lib()
    rng = np.random.default_rng(3 + len(blocks))
    M, Nd = 256, 512
    kofs = np.concatenate([[0], np.cumsum(blocks)]).astype(np.int32)
    Kp = int(kofs[-1]) * 128 + 128   # one spare block past the last group
    A, B = _codes(rng, (M, Kp)), _codes(rng, (Nd, Kp))
    sa = rng.uniform(0.05, 3.0, (Kp // 128, M)).astype(np.float32)
    sb = rng.uniform(0.05, 3.0, (Kp // 128, Nd)).astype(np.float32)
    C = m.fp8_grouped_gemm_wgrad(*(torch.from_numpy(x).cuda() for x in (A, sa, B, sb, kofs)))
    assert m.device_status() == 0
    C = C.cpu().numpy()
    for g in range(len(blocks)):
        k0, k1 = int(kofs[g]), int(kofs[g + 1])
        if k0 == k1:
            assert not C[g].any()
            continue
        ref = oracle.fp8_gemm_kscaled(A[:, k0 * 128:k1 * 128], sa[k0:k1], B[:, k0 * 128:k1 * 128], sb[k0:k1])
        assert _rowwise(C[g], ref, f"group {g}") < 1e-5


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------

def _build(sh, seed_w=1):
    m = _lib()
    cent = S.centroids(sh).cuda()
    bias = S.bias(sh).cuda()
    return m.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias,
                            lambda e: S.expert_weights(sh, e, seed=seed_w, device="cuda"), fp8=True, train=True,
                            n_groups=sh.n_groups, topk_groups=sh.topk_groups, gamma=sh.gamma)


def _cpu_weights(sh, seed_w=1):
    return lambda e: tuple(w.cpu() for w in S.expert_weights(sh, e, seed=seed_w, device="cuda"))


# Tolerance of the backward, per row against the oracle's FP64 (largest
# difference over the row's largest value). Both sides take the same E4M3
# and bf16 decisions except where a value the GPU sums in fp32 (dA, dX, the
# fp32 products fl32(g G) of the weight-gradient operand) falls on the other
# side of a bf16 or E4M3 rounding boundary than the oracle's FP64 value: that
# element then moves by one bf16 step (2^-8 of it) or one E4M3 step (up to
# 2^-3 of it), and the products downstream by that step times a weight. With
# a handful of such flips per expert the rows differ by a few 1e-3 (measured:
# at most 8e-3); a wrong scale, operand, sign or row gives order one. Bars:
# 2e-3 for h' (the forward's own bound), 2e-2 for every backward result.
TAU_BWD = 2e-2


def _backward_case(sh, seed_u=0, seed_g=0):
    m = _lib()
    layer = _build(sh)
    b0 = layer.bias.cpu().numpy().copy()
    u = S.tokens(sh, seed=seed_u)
    G = S.grad_out(sh, seed=seed_g)
    idx = torch.empty((sh.T, sh.K), dtype=torch.int32, device="cuda")
    out = layer.forward_train(u.cuda(), topk_idx=idx, update_bias=False)
    dz = torch.empty((sh.T, sh.K), dtype=torch.float32, device="cuda")
    du = layer.backward(u.cuda(), G.cuda(), dz=dz)
    assert m.device_status() == 0
    ref = oracle.layer_backward(u, layer.centroids.cpu(), b0, sh.K, _cpu_weights(sh), G, n_groups=sh.n_groups,
                                topk_groups=sh.topk_groups, fp8=True)
    assert not ref.route.near_tie.any()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref.route.topk_idx)
    return layer, out, du, dz, ref


def _check_layer_backward(sh, layer, out, du, dz, ref):
    T, K, N, I, d = sh.T, sh.K, sh.N, sh.I, sh.d
    check_bf16(out.cpu(), ref.h, tau=2e-3, what="h'")
    errs = {}
    # the forward's stored products H (bf16 of the FP8 GEMM): one rounding apart
    H = layer.train_buffer(T, "H").cpu().float().numpy()
    offs = layer.train_buffer(T, "offsets").cpu().numpy()
    for e in range(N + 1):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r0 == r1:
            continue
        inter = ref.inter[e]
        h = H[r0:r1].reshape(r1 - r0, I // 128, 2, 128)
        h1 = h[:, :, 0, :].reshape(r1 - r0, I)
        h3 = h[:, :, 1, :].reshape(r1 - r0, I)
        check_bf16(torch.from_numpy(h1), inter["Ht1"], tau=1e-3, what=f"H1[{e}]")
        check_bf16(torch.from_numpy(h3), inter["Ht3"], tau=1e-3, what=f"H3[{e}]")
        dA = layer.train_buffer(T, "dA")[r0:r1].cpu().float().numpy()
        errs[f"dA[{e}]"] = _rowwise(dA, inter["dA"], "dA")
        dX = layer.train_buffer(T, "dX")[r0:r1].cpu().float().numpy()
        errs[f"dX[{e}]"] = _rowwise(dX, inter["dX"], "dX")
    errs["du"] = _rowwise(du.cpu().float().numpy(), ref.du, "du")
    errs["dz"] = _rowwise(dz.cpu().numpy().T, ref.dz.T, "dz")
    errs["de"] = _rowwise(layer.dcentroids.cpu().numpy(), ref.de, "de")
    dw13 = layer.dw13.cpu().numpy().reshape(N + 1, I // 128, 2, 128, d)
    dw1 = dw13[:, :, 0].reshape(N + 1, I, d)
    dw3 = dw13[:, :, 1].reshape(N + 1, I, d)
    dw2 = layer.dw2.cpu().numpy()
    for e in range(N + 1):
        errs[f"dw1[{e}]"] = _rowwise(dw1[e], ref.dw1[e], "dw1")
        errs[f"dw3[{e}]"] = _rowwise(dw3[e], ref.dw3[e], "dw3")
        errs[f"dw2[{e}]"] = _rowwise(dw2[e], ref.dw2[e], "dw2")
    worst = max(errs, key=errs.get)
    print("backward errors: worst", worst, errs[worst], {k: round(v, 5) for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v < TAU_BWD}
    assert not bad, bad


def test_layer_backward_small():
    sh = S.LayerShape(T=200, d=256, N=8, K=2, I=256, name="bwd-small")
    _check_layer_backward(sh, *_backward_case(sh))


def test_layer_backward_ragged_groups_and_top4():
    """Experts of ~150-300 rows (several 128-row weight-gradient blocks, ragged
    tails), d = 512, top-4 of 8."""
    sh = S.LayerShape(T=301, d=512, N=8, K=4, I=256, name="bwd-ragged")
    _check_layer_backward(sh, *_backward_case(sh, seed_u=3, seed_g=4))


def test_layer_backward_group_limited():
    sh = S.LayerShape(T=96, d=256, N=16, K=4, I=256, n_groups=4, topk_groups=2, name="bwd-groups")
    _check_layer_backward(sh, *_backward_case(sh, seed_u=5, seed_g=6))


def test_layer_backward_kblock_offsets_bit_exact():
    sh = S.LayerShape(T=300, d=256, N=8, K=2, I=256, name="bwd-kofs")
    layer, out, du, dz, ref = _backward_case(sh)
    offs = layer.train_buffer(sh.T, "offsets").cpu().numpy()
    kofs = layer.train_buffer(sh.T, "kofs").cpu().numpy()
    n = np.diff(offs.astype(np.int64))
    np.testing.assert_array_equal(kofs, np.concatenate([[0], np.cumsum((n + 127) // 128)]))
    np.testing.assert_array_equal(offs[:sh.N + 1], ref.offsets)


def test_layer_backward_empty_batch():
    m = _lib()
    sh = S.LayerShape(T=0, d=256, N=8, K=2, I=256, name="bwd-empty")
    layer = _build(S.LayerShape(T=16, d=256, N=8, K=2, I=256))
    layer.dw13.fill_(1.0)
    layer.dw2.fill_(1.0)
    layer.dcentroids.fill_(1.0)
    u = torch.empty((0, sh.d), dtype=torch.bfloat16, device="cuda")
    layer.forward_train(u, update_bias=False)
    du = layer.backward(u, u)
    assert du.shape == (0, sh.d) and m.device_status() == 0
    assert not layer.dw13.any() and not layer.dw2.any() and not layer.dcentroids.any()


def test_layer_backward_experts_without_tokens_get_zero_gradients():
    """A bias that shuts experts out leaves them no rows: their weight
    gradients are exactly zero, the others match the oracle."""
    m = _lib()
    sh = S.LayerShape(T=128, d=256, N=8, K=2, I=256, name="bwd-idle")
    layer = _build(sh)
    layer.bias[5:].fill_(-1.0e4)   # experts 5, 6, 7 never chosen
    b0 = layer.bias.cpu().numpy().copy()
    u, G = S.tokens(sh), S.grad_out(sh)
    out = layer.forward_train(u.cuda(), update_bias=False)
    du = layer.backward(u.cuda(), G.cuda())
    assert m.device_status() == 0
    assert not layer.dw13[5:8].any() and not layer.dw2[5:8].any() and not layer.dcentroids[5:8].any()
    ref = oracle.layer_backward(u, layer.centroids.cpu(), b0, sh.K, _cpu_weights(sh), G, fp8=True)
    assert _rowwise(du.cpu().float().numpy(), ref.du, "du") < TAU_BWD
    for e in (0, sh.N):
        assert _rowwise(layer.dw2[e].cpu().numpy(), ref.dw2[e], "dw2") < TAU_BWD


def test_training_steps_match_the_oracle():
    """Two SGD steps: the bias bit-exact after each, the masters' moves
    lr * dW within the backward's tolerance, and the second step's h' (from
    re-quantised weights and moved centroids) within the forward's. The step
    (lr |dW| about 1 % of |w|) keeps the two sides' second steps on weights
    that agree to ~1e-4, as the first step's gradients agree to ~1e-2."""
    m = _lib()
    sh = S.LayerShape(T=160, d=256, N=8, K=2, I=256, name="train")
    layer = _build(sh)
    lr = 2e-4
    N, I, d = sh.N, sh.I, sh.d
    ws = [tuple(w.cpu().float().numpy() for w in S.expert_weights(sh, e, seed=1, device="cuda")) for e in range(N + 1)]
    masters = {"w1": np.stack([w[0] for w in ws]), "w3": np.stack([w[1] for w in ws]),
               "w2": np.stack([w[2] for w in ws]), "e": layer.centroids.cpu().numpy().copy()}
    bias = layer.bias.cpu().numpy().copy()
    for step in range(2):
        u, G = S.tokens(sh, seed=10 + step), S.grad_out(sh, seed=20 + step)
        w13_before = layer.w13_master.clone()
        e_before = layer.centroids.clone()
        out, du = layer.train_step(u.cuda(), G.cuda(), lr)
        assert m.device_status() == 0
        new, bias_new, bw = oracle.train_step(u, masters, bias, sh.K, G, lr, sh.gamma)
        check_bf16(out.cpu(), bw.h, tau=2e-3, what=f"h' step {step}")
        np.testing.assert_array_equal(layer.bias.cpu().numpy(), bias_new)
        moved = (layer.w13_master - w13_before).cpu().numpy().reshape(N + 1, I // 128, 2, 128, d)
        exp1 = (new["w1"] - masters["w1"]).reshape(N + 1, I // 128, 128, d)
        for e in range(N + 1):
            assert _rowwise(moved[e, :, 0].reshape(I, d), exp1[e].reshape(I, d), f"w1 move {step}") < TAU_BWD, \
                (step, e)
        de = (layer.centroids - e_before).cpu().numpy()
        assert _rowwise(de, new["e"] - masters["e"], "centroid move") < TAU_BWD
        masters, bias = new, bias_new
    # the layer's FP8 weights hold its own masters: each code within half an E4M3
    # step of master / scale (3 mantissa bits: 2^-4 of the value, or 2^-10 below
    # the normal range), and the transposed copy is the same codes
    vals = _vals()
    for e in (0, N):
        w = layer.w2_master[e].cpu().numpy().astype(np.float64)
        sc = np.repeat(np.repeat(layer.w2_scales[e].cpu().numpy().astype(np.float64), 128, 0), 128, 1)
        q = layer.w2[e].cpu().numpy()
        x = w / sc
        assert np.all(np.abs(vals[q] - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) * 1.0000001)
        np.testing.assert_array_equal(layer.w2t[e].cpu().numpy(), q.T)


def test_training_step_graph_replay_matches_eager():
    """The training step captured in a CUDA graph and replayed on two batches
    leaves the same bits as two eager steps: h', du, masters, FP8 weights and
    their transposed copies, scales, centroids, bias."""
    m = _lib()
    sh = S.LayerShape(T=128, d=256, N=8, K=2, I=256, name="train-graph")
    eager, graphed = _build(sh), _build(sh)
    lr = 1e-3
    u = torch.empty((sh.T, sh.d), dtype=torch.bfloat16, device="cuda")
    G = torch.empty_like(u)
    g = graphed.capture_train(u, G, lr)
    for step in range(2):
        ub, Gb = S.tokens(sh, seed=50 + step).cuda(), S.grad_out(sh, seed=60 + step).cuda()
        out_e, du_e = eager.train_step(ub, Gb, lr)
        u.copy_(ub)
        G.copy_(Gb)
        out_g, du_g = g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16)), step
        assert torch.equal(du_g.view(torch.int16), du_e.view(torch.int16)), step
        for name in ("w13_master", "w2_master", "w13", "w13_scales", "w2", "w2_scales", "w13t", "w2t", "centroids",
                     "bias"):
            a, b = getattr(graphed, name), getattr(eager, name)
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (step, name)
    assert m.device_status() == 0
