"""Parity of each C-ABI entry point against the FP64 oracle, on the GPU.

Inputs come from the seeded generator; where a kernel consumes another stage's
output, the test feeds both sides the same oracle-made (or generated) values.
Integer/byte/index results must match bit for bit; floating outputs follow the
rules in tests/helpers.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import check_bf16, check_fp8_codes, e4m3_values

pytestmark = pytest.mark.gpu

M = None


def lib():
    global M
    if M is None:
        import mixture_experts_layer_90_b300 as m
        M = m
    return M


def cuda(x):
    return torch.as_tensor(x).cuda()


def status_ok():
    assert lib().device_status() == 0


def bf16(shape, std, *name, outliers=0):
    x = S.normal(shape, std, S.key(0, *name), dtype=torch.float32)
    if outliers:
        pos = S.choose_positions(x.numel(), outliers, S.key(0, *name, "outliers"))
        x.view(-1)[pos] *= 100.0
    return x.to(torch.bfloat16)


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 640), (300, 1024), (4096, 7168)])
def test_quant_1x128_bit_exact(rows, cols):
    x = bf16((rows, cols), 1.0, "q1", rows, cols, outliers=max(1, rows * cols // 1000))
    q, s = lib().fp8_quant_1x128(cuda(x))
    qo, so = oracle.quant_1x128(x)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so.T)
    status_ok()


def test_quant_1x128_strided_rows_and_zero_tiles():
    x = bf16((64, 512), 1.0, "q1s")
    x[5] = 0.0
    x[7, 128:256] = -0.0
    big = torch.zeros((64, 768), dtype=torch.bfloat16)
    big[:, :512] = x
    q, s = lib().fp8_quant_1x128(cuda(big)[:, :512])
    qo, so = oracle.quant_1x128(x)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so.T)


@pytest.mark.parametrize("rows,cols", [(128, 128), (300, 384), (4096, 7168)])
def test_quant_128x128_bit_exact(rows, cols):
    w = bf16((rows, cols), 0.02, "q128", rows, cols, outliers=max(1, rows * cols // 10000))
    q, s = lib().fp8_quant_128x128(cuda(w))
    qo, so = oracle.quant_128x128(w)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so)
    status_ok()


def test_e4m3_conversion_every_bf16_value():
    """Every bf16 value of magnitude <= 448 (both signs), quantised with the
    tile scale pinned to exactly 1, converts as the oracle's encoder."""
    bits = np.arange(0, 0x43E1, dtype=np.uint32)          # +0 .. 448 as bf16 bit patterns
    v = (bits << 16).view(np.float32)
    v = v[np.abs(v) <= 448.0]
    v = np.concatenate([v, -v])
    pad = (-v.size) % 127
    v = np.concatenate([v, np.zeros(pad, np.float32)]).reshape(-1, 127)
    v = np.concatenate([np.full((v.shape[0], 1), 448.0, np.float32), v], axis=1)   # scale = 448/448 = 1
    x = torch.from_numpy(v).to(torch.bfloat16)
    q, s = lib().fp8_quant_1x128(cuda(x))
    assert np.all(s.cpu().numpy() == 1.0)
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.e4m3_encode(v))


def test_quant_1x128_every_bf16_value_under_many_scales():
    """The quantiser forms x / scale by reciprocal where that cannot change the
    code (and divides elsewhere): every bf16 value up to a tile's amax, for amax
    in many binades (tiny ones whose scale is below the smallest normal float
    included), must give the oracle's codes, which come from IEEE divisions."""
    rng = np.random.Generator(np.random.PCG64(9))
    amax_bits = np.concatenate([rng.integers(0x0080, 0x7F80, 24), [0x43E0, 0x3F80, 0x0200, 0x0480, 0x0500, 0x7F7F]])
    rows = []
    for ab in amax_bits.astype(np.uint32):
        amax = np.array([ab << 16], np.uint32).view(np.float32)[0]
        g = (np.arange(0, ab + 1, dtype=np.uint32) << 16).view(np.float32)
        g = np.concatenate([g, -g])
        g = np.concatenate([g, np.zeros((-g.size) % 127, np.float32)]).reshape(-1, 127)
        rows.append(np.concatenate([np.full((g.shape[0], 1), amax, np.float32), g], axis=1))
    v = np.concatenate(rows)
    x = torch.from_numpy(v).to(torch.bfloat16)
    q, s = lib().fp8_quant_1x128(cuda(x))
    qo, so = oracle.quant_1x128(x)
    np.testing.assert_array_equal(s.cpu().numpy(), so.T)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    status_ok()


# --------------------------------------------------------------------------
# FP8 GEMMs
# --------------------------------------------------------------------------

def _weights_fp8(G, Nd, Kd, name, std=0.05):
    qs, ss = [], []
    for g in range(G):
        w = bf16((Nd, Kd), std, name, g, Nd, Kd)
        q, s = oracle.quant_128x128(w)
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)


def _acts_fp8(Mr, Kd, name, outliers=0):
    a = bf16((Mr, Kd), 1.0, name, Mr, Kd, outliers=outliers)
    return oracle.quant_1x128(a)


@pytest.mark.parametrize("offsets", [[0, 300], [0, 130, 130, 400, 401], [0, 0, 1, 129, 256, 517]])
@pytest.mark.parametrize("Nd,Kd", [(256, 128), (512, 384)])
def test_fp8_grouped_gemm_bf16_out(offsets, Nd, Kd):
    G = len(offsets) - 1
    Mr = offsets[-1] + 3                       # trailing rows that belong to no group
    qa, sa = _acts_fp8(Mr, Kd, "ga", outliers=Mr * Kd // 1000)
    qb, sb = _weights_fp8(G, Nd, Kd, "gb")
    C = torch.full((Mr, Nd), float("nan"), dtype=torch.bfloat16).cuda()
    lib().fp8_grouped_gemm(cuda(qa), cuda(np.ascontiguousarray(sa.T)), cuda(qb), cuda(sb),
                           cuda(np.array(offsets, np.int32)), lib().MOE_EPI_BF16, C=C)
    status_ok()
    Cg = C.cpu()
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        ref = oracle.fp8_gemm(qa[r0:r1], sa[r0:r1], qb[g], sb[g])
        tau = check_bf16(Cg[r0:r1], ref, what=f"group {g}")
        print(f"group {g}: achieved tau {tau:.2e}")
    assert torch.isnan(Cg[offsets[-1]:].float()).all()      # rows past the last group untouched


def _swiglu_ref(qa, sa, qb, sb):
    C = oracle.fp8_gemm(qa, sa, qb, sb)
    Nd = qb.shape[0]
    j = np.arange(Nd // 2)
    gate = (j // 128) * 256 + j % 128
    return C[:, gate], C[:, gate + 128]


@pytest.mark.parametrize("offsets", [[0, 200], [0, 1, 1, 257, 300]])
def test_fp8_grouped_gemm_swiglu_fp8_out(offsets):
    G, Nd, Kd = len(offsets) - 1, 512, 512
    Mr = offsets[-1]
    qa, sa = _acts_fp8(Mr, Kd, "sa", outliers=50)
    qb, sb = _weights_fp8(G, Nd, Kd, "sb", std=1.0 / math.sqrt(Kd))
    C, cs = lib().fp8_grouped_gemm(cuda(qa), cuda(np.ascontiguousarray(sa.T)), cuda(qb), cuda(sb),
                                   cuda(np.array(offsets, np.int32)), lib().MOE_EPI_SWIGLU_FP8)
    status_ok()
    C, cs = C.cpu().numpy(), cs.cpu().numpy().T
    flips = 0
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        h1, h3 = _swiglu_ref(qa[r0:r1], sa[r0:r1], qb[g], sb[g])
        q, s, dist, v = oracle.swiglu_quant(h1, h3)
        np.testing.assert_allclose(cs[r0:r1], s, rtol=1e-5)
        flips += check_fp8_codes(C[r0:r1], q, dist, v, what=f"group {g}")
    assert flips <= C.size * 1e-3


def test_fp8_gemm_dense_full_size_sampled_rows():
    """The dense 4096 x 7168 x 4096 block-scaled GEMM with 0.1% x100 outliers in
    A (the FP8-GEMM workload): the oracle computes 64 sampled output rows."""
    cfg = S.GEMM_V3
    a, b = S.gemm_operands(cfg["M"], cfg["K"], cfg["N"])
    qa, sa = lib().fp8_quant_1x128(cuda(a))
    qb, sb = lib().fp8_quant_128x128(cuda(b))
    C = lib().fp8_grouped_gemm(qa, sa, qb[None], sb[None], cuda(np.array([0, cfg["M"]], np.int32)))
    status_ok()
    # the oracle quantises the same bf16 inputs itself
    qa_o, sa_o = oracle.quant_1x128(a)
    qb_o, sb_o = oracle.quant_128x128(b)
    rng = np.random.Generator(np.random.PCG64(4))
    rows = np.unique(np.concatenate([[0, 1, 127, 128, cfg["M"] - 1], rng.choice(cfg["M"], 59, replace=False)]))
    ref = oracle.fp8_gemm(qa_o[rows], sa_o[rows], qb_o, sb_o)
    got = C[torch.as_tensor(rows).cuda()].cpu()
    tau = check_bf16(got, ref, what="dense fp8 gemm")
    print(f"dense FP8 GEMM: achieved tau {tau:.2e}")


# --------------------------------------------------------------------------
# bf16 GEMMs
# --------------------------------------------------------------------------

@pytest.mark.parametrize("epi", ["bf16", "swiglu", "f32"])
def test_bf16_grouped_gemm(epi):
    offsets = [0, 100, 100, 229, 230]
    G, Nd, Kd = 4, 512, 320
    Mr = offsets[-1]
    a = bf16((Mr, Kd), 1.0, "ba")
    b = torch.stack([bf16((Nd, Kd), 1.0 / math.sqrt(Kd), "bb", g) for g in range(G)])
    e = {"bf16": lib().MOE_EPI_BF16, "swiglu": lib().MOE_EPI_SWIGLU_BF16, "f32": lib().MOE_EPI_F32}[epi]
    C = lib().bf16_grouped_gemm(cuda(a), cuda(b), cuda(np.array(offsets, np.int32)), e).cpu()
    status_ok()
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        ref = oracle.bf16_gemm(a[r0:r1], b[g])
        if epi == "bf16":
            check_bf16(C[r0:r1], ref, tau=1e-5)
        elif epi == "f32":
            np.testing.assert_allclose(C[r0:r1].numpy(), ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())
        else:
            j = np.arange(Nd // 2)
            gate = (j // 128) * 256 + j % 128
            a_ref = oracle.swiglu(ref[:, gate], ref[:, gate + 128])
            check_bf16(C[r0:r1], a_ref, tau=1e-5)


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

from helpers import ROUTE_DELTA


def _route_case(T, d, N, f32, zero_bias=False, seed=0):
    u = S.normal((T, d), 1.0, S.key(seed, "route-u", T, d))
    e = S.normal((N, d), 1.0 / math.sqrt(d), S.key(seed, "route-e", N, d),
                 dtype=torch.float32 if f32 else torch.bfloat16)
    b = torch.zeros(N) if zero_bias else S.uniform((N,), -0.01, 0.01, S.key(seed, "route-b", N))
    return u, e, b


def _check_route(u, e, b, K, n_groups=1, topk_groups=1):
    T = u.shape[0]
    idx, gates, loads, scores = lib().moe_route(cuda(u), cuda(e), cuda(b), K, n_groups, topk_groups,
                                                want_scores=True)
    status_ok()
    idx, gates, loads, scores = idx.cpu().numpy(), gates.cpu().numpy(), loads.cpu().numpy(), scores.cpu().numpy()
    r = oracle.route(u, e, b, K, n_groups, topk_groups, delta=ROUTE_DELTA, want_scores=True)
    # the fp32 affinities and the certification margin
    s_err = np.max(np.abs(scores - r.scores))
    # keys differ from the oracle's by at most s_err plus the fp32 rounding of s + b;
    # two such errors must fit inside the certified gap
    assert 2 * (s_err + 2 ** -23) < ROUTE_DELTA, f"affinity error {s_err:.2e} too large for the certified gap"
    same = np.all(idx == r.topk_idx, axis=1)
    assert np.all(same | r.near_tie), "a token with a certified gap was routed differently"
    # tokens near a tie: the GPU's set must be as good as the oracle's within delta
    key = r.scores + b.double().numpy()[None, :]
    for t in np.nonzero(~same)[0]:
        kth = np.sort(key[t, r.topk_idx[t]])[0]
        assert np.all(key[t, idx[t]] >= kth - ROUTE_DELTA)
    assert np.all(np.diff(idx, axis=1) > 0)
    # gates from raw affinities, normalised over the chosen experts
    np.testing.assert_allclose(gates[same], r.gates[same], rtol=2e-6, atol=0)
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=0, atol=2e-6)
    np.testing.assert_array_equal(loads, np.bincount(idx.ravel(), minlength=e.shape[0]))
    if same.all():
        np.testing.assert_array_equal(loads, r.loads)
    return idx, r, int((~same).sum()), int(r.near_tie.sum())


def test_route_tiny_bf16_centroids():
    u, e, b = _route_case(128, 256, 16, f32=False, zero_bias=True)
    _check_route(u, e, b, K=4)


@pytest.mark.parametrize("T,d,N,K", [(1000, 1024, 256, 8), (33, 512, 64, 6), (257, 2048, 1024, 16)])
def test_route_fp32_centroids(T, d, N, K):
    u, e, b = _route_case(T, d, N, f32=True)
    _check_route(u, e, b, K)


def test_route_group_limited():
    u, e, b = _route_case(700, 512, 256, f32=True)
    idx, r, _, _ = _check_route(u, e, b, K=8, n_groups=8, topk_groups=4)
    assert np.all(np.array([len(set(row // 32)) for row in idx]) <= 4)


def test_route_forced_bias():
    u, e, b = _route_case(300, 512, 64, f32=True)
    b = b.clone()
    b[[1, 9, 33, 63]] = 10.0
    b[[0, 2]] = -10.0
    idx, gates, loads, _ = lib().moe_route(cuda(u), cuda(e), cuda(b), 6)
    loads = loads.cpu().numpy()
    assert np.all(loads[[1, 9, 33, 63]] == 300) and loads[0] == 0 and loads[2] == 0
    assert loads.sum() == 300 * 6


@pytest.mark.parametrize("f32,n_groups", [(True, 1), (False, 1), (True, 8)])
def test_route_prepared_is_bit_identical(f32, n_groups):
    """moe_route_prepare_centroids + moe_route_prepared give exactly what
    moe_route gives, on two calls that reuse one prepared operand."""
    m = lib()
    N, K = (256, 8) if n_groups > 1 else (64, 6)
    u, e, b = _route_case(300, 512, N, f32=f32)
    prepared = m.moe_route_prepare_centroids(cuda(e))
    cdt = m.MOE_DTYPE_F32 if f32 else m.MOE_DTYPE_BF16
    for seed in (0, 1):
        uu = u if seed == 0 else S.normal(u.shape, 1.0, S.key(seed, "route-u2"))
        a = m.moe_route(cuda(uu), cuda(e), cuda(b), K, n_groups, 4 if n_groups > 1 else 1, want_scores=True)
        p = m.moe_route_prepared(cuda(uu), prepared, cdt, N, cuda(b), K, n_groups, 4 if n_groups > 1 else 1,
                                 want_scores=True)
        status_ok()
        for x, y in zip(a, p):
            assert torch.equal(x, y)


def test_route_full_size():
    """The route+dispatch workload: T=16384, d=7168, 256 fp32 centroids, top-8."""
    sh = S.ROUTE_V3
    u = S.tokens(sh)
    e = S.centroids(sh)
    b = S.bias(sh)
    _, r, n_diff, n_near = _check_route(u, e, b, K=sh.K)
    print(f"route full size: {n_near} tokens within the certified gap, {n_diff} routed differently")


# --------------------------------------------------------------------------
# permutation
# --------------------------------------------------------------------------

def _rand_topk(T, N, K, seed=0):
    h = S.bits(S.key(seed, "topk", T, N, K), 0, T * N).view(T, N)
    return torch.sort(torch.argsort(h, dim=1)[:, :K], dim=1).values.to(torch.int32).numpy()


@pytest.mark.parametrize("T,d,N,K,fp8,shared", [(1, 128, 4, 2, False, False), (1000, 512, 16, 4, False, True),
                                                 (333, 640, 256, 8, True, True), (64, 256, 1024, 16, True, False),
                                                 # widths that leave part of the warp's 512-column step idle
                                                 (77, 384, 8, 3, False, True), (129, 896, 64, 6, False, False),
                                                 (50, 128, 4, 2, True, True), (91, 1152, 32, 5, True, False),
                                                 # either side of the single-block path's limit (8192 pairs,
                                                 # 256 experts): the last one-block batch, then ragged
                                                 # multi-block batches just past the pair and expert limits
                                                 (1024, 256, 256, 8, True, True), (1025, 256, 256, 8, False, True),
                                                 (1500, 128, 32, 6, False, False), (100, 128, 257, 8, True, True)])
def test_permute_bit_exact(T, d, N, K, fp8, shared):
    x = bf16((T, d), 1.0, "px", T, d)
    idx = _rand_topk(T, N, K)
    dt = lib().MOE_DTYPE_E4M3 if fp8 else lib().MOE_DTYPE_BF16
    off, perm, dest, xp, xs = lib().moe_permute(cuda(x), cuda(idx), N, dt, with_shared=shared)
    status_ok()
    off_o, perm_o, dest_o = oracle.permute(idx, N)
    exp_off = np.concatenate([off_o, [off_o[-1] + T]]) if shared else off_o
    np.testing.assert_array_equal(off.cpu().numpy(), exp_off)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_o)
    np.testing.assert_array_equal(dest.cpu().numpy(), dest_o)
    src = np.concatenate([perm_o, np.arange(T)]) if shared else perm_o
    if fp8:
        q, s = oracle.quant_1x128(x)
        np.testing.assert_array_equal(xp.cpu().numpy(), q[src])
        np.testing.assert_array_equal(xs.cpu().numpy(), s[src].T)
    else:
        np.testing.assert_array_equal(xp.cpu().view(torch.int16).numpy(), x.view(torch.int16).numpy()[src])


def test_permute_full_size_bf16():
    sh = S.ROUTE_V3
    T, d, N, K = sh.T, sh.d, sh.N, sh.K
    x = cuda(S.tokens(sh))
    idx = _rand_topk(T, N, K, seed=1)
    off, perm, dest, xp, _ = lib().moe_permute(x, cuda(idx), N)
    status_ok()
    off_o, perm_o, dest_o = oracle.permute(idx, N)
    np.testing.assert_array_equal(off.cpu().numpy(), off_o)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_o)
    np.testing.assert_array_equal(dest.cpu().numpy(), dest_o)
    _assert_rows_equal(xp, x, perm_o)


def _assert_rows_equal(xp, x, src, chunk=8192):
    """Every permuted row equals its source row, byte for byte (compared on the
    device, `chunk` rows at a time)."""
    src = torch.as_tensor(src).cuda().long()
    assert xp.shape[0] == src.numel()
    for r0 in range(0, src.numel(), chunk):
        r1 = min(src.numel(), r0 + chunk)
        assert torch.equal(xp[r0:r1].view(torch.int16), x[src[r0:r1]].view(torch.int16)), f"rows {r0}..{r1}"


def test_route_dispatch_full_size_composition():
    """The route + dispatch workload end to end at T=16384, d=7168, 256 fp32
    centroids, top-8: moe_route's own output feeds moe_permute (bf16 rows) and
    moe_bias_update. Routing is checked against the oracle with the certified-gap
    rule; the permutation (offsets, perm_token, dest_row, every row's bytes) and
    the updated bias are checked bit-exactly against the oracle run on the GPU's
    selection."""
    m = lib()
    sh = S.ROUTE_V3
    T, d, N, K = sh.T, sh.d, sh.N, sh.K
    u, e, b = S.tokens(sh), S.centroids(sh), S.bias(sh)
    x = cuda(u)
    idx_t, gates, loads_t, _ = m.moe_route(x, cuda(e), cuda(b), K)
    off, perm, dest, xp, _ = m.moe_permute(x, idx_t, N)
    bias_t = cuda(b.clone())
    m.moe_bias_update(bias_t, loads_t, T, K, sh.gamma)
    status_ok()
    idx, loads = idx_t.cpu().numpy(), loads_t.cpu().numpy()
    r = oracle.route(u, e, b, K, delta=ROUTE_DELTA)
    same = np.all(idx == r.topk_idx, axis=1)
    assert np.all(same | r.near_tie), "a token with a certified gap was routed differently"
    np.testing.assert_array_equal(loads, np.bincount(idx.ravel(), minlength=N))
    if same.all():
        np.testing.assert_array_equal(loads, r.loads)
    np.testing.assert_allclose(gates.cpu().numpy()[same], r.gates[same], rtol=2e-6, atol=0)
    off_o, perm_o, dest_o = oracle.permute(idx, N)
    np.testing.assert_array_equal(off.cpu().numpy(), off_o)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_o)
    np.testing.assert_array_equal(dest.cpu().numpy(), dest_o)
    _assert_rows_equal(xp, x, perm_o)
    np.testing.assert_array_equal(bias_t.cpu().numpy(), oracle.bias_update(b.numpy(), loads, T, K, sh.gamma))
    print(f"route+dispatch full size: {int(r.near_tie.sum())} near-tie tokens, {int((~same).sum())} routed "
          f"differently; loads max {loads.max()}, min {loads.min()}")


# --------------------------------------------------------------------------
# combine, bias update
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,d,K,shared", [(1, 256, 1, True), (300, 512, 8, True), (77, 384, 4, False)])
def test_combine(T, d, K, shared):
    N = 32
    idx = _rand_topk(T, N, K, seed=2)
    _, _, dest = oracle.permute(idx, N)
    R = T * K + T
    u = bf16((T, d), 1.0, "cu", T, d)
    y = bf16((R, d), 0.5, "cy", R, d)
    g = S.uniform((T, K), 0.05, 1.0, S.key(0, "cg", T, K))
    g = (g / g.sum(1, keepdim=True)).float()
    ys = y[T * K:] if shared else None
    out = lib().moe_combine(cuda(u), cuda(ys) if shared else None, cuda(y), cuda(g), cuda(dest))
    status_ok()
    ref = oracle.combine(u, ys, y, g.double().numpy(), dest)
    check_bf16(out.cpu(), ref, tau=1e-6, what="combine")


def test_combine_zero_experts_returns_u():
    T, d, K = 50, 256, 4
    u = bf16((T, d), 1.0, "cz")
    y = torch.zeros((T * K + T, d), dtype=torch.bfloat16)
    dest = oracle.permute(_rand_topk(T, 16, K, seed=3), 16)[2]
    g = torch.full((T, K), 0.25)
    out = lib().moe_combine(cuda(u), cuda(y[T * K:]), cuda(y), cuda(g), cuda(dest)).cpu()
    assert torch.equal(out.view(torch.int16), u.view(torch.int16))


@pytest.mark.parametrize("T,K,N", [(10, 4, 8), (16384, 8, 256), (7, 3, 5)])
def test_bias_update_bit_exact(T, K, N):
    rng = np.random.Generator(np.random.PCG64(T))
    loads = rng.multinomial(T * K, np.ones(N) / N).astype(np.int32)
    loads[0] = (T * K) // N if (T * K) % N == 0 else loads[0]
    b = S.uniform((N,), -0.01, 0.01, S.key(0, "bu", N)).numpy()
    bt = cuda(b.copy())
    lib().moe_bias_update(bt, cuda(loads), T, K, 1e-3)
    np.testing.assert_array_equal(bt.cpu().numpy(), oracle.bias_update(b, loads, T, K, 1e-3))


# --------------------------------------------------------------------------
# sequence-wise balance statistics
# --------------------------------------------------------------------------

def _check_balance(u, e, b, K, seq_len, n_groups=1, topk_groups=1):
    m = lib()
    T = u.shape[0]
    idx, _, _, scores = m.moe_route(cuda(u), cuda(e), cuda(b), K, n_groups, topk_groups, want_scores=True)
    loads, prob, stat = m.moe_route_balance_stats(scores, idx, seq_len)
    loads2, prob2, stat2 = m.moe_route_balance_stats(scores, idx, seq_len)
    status_ok()
    # fixed summation order: a second call gives the same bits
    assert torch.equal(loads, loads2) and torch.equal(prob, prob2) and torch.equal(stat, stat2)
    r = oracle.route(u, e, b, K, n_groups, topk_groups, delta=ROUTE_DELTA, want_scores=True)
    idx_g = idx.cpu().numpy()
    same = np.all(idx_g == r.topk_idx, axis=1)
    assert np.all(same | r.near_tie)
    ol, op, os_ = oracle.seq_balance(r.scores, r.topk_idx, K, seq_len)
    if same.all():
        np.testing.assert_array_equal(loads.cpu().numpy(), ol)
    else:
        # near-tie tokens routed to another equally good set: loads follow the GPU's selection
        np.testing.assert_array_equal(loads.cpu().numpy(), oracle.seq_balance(r.scores, idx_g, K, seq_len)[0])
    # P from fp32 affinities (|s - s_oracle| <= 5e-6) summed in fp32
    np.testing.assert_allclose(prob.cpu().numpy(), op, rtol=2e-5, atol=1e-7)
    gl = loads.cpu().numpy().astype(np.float64)
    lens = np.array([min(seq_len, T - t0) for t0 in range(0, T, seq_len)], np.float64)
    ref_stat = ((e.shape[0] * gl / (K * lens[:, None])) * op).sum(axis=1)
    np.testing.assert_allclose(stat.cpu().numpy(), ref_stat, rtol=2e-5)
    if same.all():
        np.testing.assert_allclose(stat.cpu().numpy(), os_, rtol=2e-5)
    return stat.cpu().numpy()


@pytest.mark.parametrize("T,d,N,K,seq_len", [(1000, 512, 64, 6, 128), (77, 256, 16, 4, 1000), (300, 512, 256, 8, 64)])
def test_balance_stats(T, d, N, K, seq_len):
    u, e, b = _route_case(T, d, N, f32=True)
    _check_balance(u, e, b, K, seq_len)


def test_balance_stats_group_limited():
    u, e, b = _route_case(512, 512, 256, f32=True)
    _check_balance(u, e, b, 8, 200, n_groups=8, topk_groups=4)


def test_balance_stats_closed_forms():
    """Equal affinities give 1 whatever the routing; every token sending its
    pairs to experts 0..K-1 with all affinity there gives N/K."""
    m = lib()
    T, N, K = 256, 32, 4
    idx = torch.tensor(_rand_topk(T, N, K, seed=7))
    sc = torch.full((T, N), 0.3)
    _, prob, stat = m.moe_route_balance_stats(cuda(sc), cuda(idx), 100)
    status_ok()
    np.testing.assert_allclose(prob.cpu().numpy(), 1.0 / N, rtol=1e-6)
    np.testing.assert_allclose(stat.cpu().numpy(), 1.0, rtol=1e-6)
    idx = torch.arange(K, dtype=torch.int32).repeat(T, 1)
    sc = torch.zeros((T, N))
    sc[:, :K] = 0.7
    loads, _, stat = m.moe_route_balance_stats(cuda(sc), cuda(idx), T)
    status_ok()
    assert loads[0, :K].eq(T).all() and loads[0, K:].eq(0).all()
    np.testing.assert_allclose(stat.cpu().numpy(), N / K, rtol=1e-6)


def test_balance_stats_full_size():
    """The route + dispatch workload (T=16384, 256 experts, top-8) in sequences of 4096 tokens."""
    sh = S.ROUTE_V3
    stat = _check_balance(S.tokens(sh), S.centroids(sh), S.bias(sh), sh.K, 4096)
    print(f"sequence-wise balance statistic per sequence: {stat}")
