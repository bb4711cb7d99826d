"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- an independent library's rounding, exhaustive sorting,
closed forms and special cases, and the invariants the pages state.

Page citations: "Prox: Training-Free FFN Activation Sparsity via Approximate
Intermediate-Channel Salience in LLMs", Abstract (two stages, shared mask from
magnitude ranking, exact Stage 2); "PrunePath: Towards Highly Structured
Sparse Language Models", Sec. 2.1 Eq. (1) (SwiGLU FFN) and Sec. 2.2 Eq. (2)
(activating every block after a channel permutation is the identity).
"""
import math
import os

import numpy as np
import pytest
import torch

from free_swiglu_ffn_prox_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(a) -> np.ndarray:
    return synth.bits(torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


# ------------------------------------------------------------------ formats
def test_fp16_decode_matches_numpy_for_every_pattern(oracle_mod):
    pats = np.arange(0, 1 << 16, 97, dtype=np.uint32).astype(np.uint16)
    pats = np.concatenate([pats, np.array([0, 1, 0x3FF, 0x400, 0x7BFF, 0x7C00, 0x8001, 0xFBFF],
                                          dtype=np.uint16)])
    finite = (pats & 0x7C00) != 0x7C00
    ours = oracle_mod.fp16_to_double(pats[finite])
    ref = pats[finite].view(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_bf16_decode_matches_torch(oracle_mod):
    pats = np.arange(0, 1 << 16, 61, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle_mod.bf16_bits_to_f64(pats), ref)
    assert np.array_equal(oracle_mod.bf16_to_double(pats[:300]), ref[:300])


def test_fp16_rounding_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * np.float32(0.01),
        rng.standard_normal(500).astype(np.float32) * np.float32(3e-6),   # subnormal range
        rng.standard_normal(500).astype(np.float32) * np.float32(2e4),
    ])
    ours = oracle_mod.round_to_fp16(vals)
    ref = vals.astype(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_fp16_rounding_golden_ieee_cases(oracle_mod):
    """Hand-derived binary16 round-to-nearest-even cases (IEEE 754)."""
    rows = []
    with open(os.path.join(GOLDEN, "fp16_rne_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, b = line.split()
                rows.append((float.fromhex(a), float(b) if b != "inf" else math.inf))
    for inp, want in rows:
        got = oracle_mod.round_to_fp16(np.float32(inp))
        assert got == want, (inp, got, want)


def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(3000) * 3).astype(np.float32)
    v[:10] = [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -2.5, 3e-39, 1e38, 255.5, 256.5]
    ref = synth.bits(torch.from_numpy(v).to(torch.bfloat16))
    assert np.array_equal(oracle_mod.double_to_bf16(v.astype(np.float64)), ref)


def test_silu_closed_forms(oracle_mod):
    assert oracle_mod.silu(0.0) == 0.0
    ln3 = math.log(3.0)
    assert abs(oracle_mod.silu(ln3) - 0.75 * ln3) < 1e-15   # sigma(ln 3) = 3/4
    assert oracle_mod.silu(40.0) == 40.0                     # sigma(40) rounds to 1
    for z in (-7.5, -1.0, 0.3, 2.0, 11.0):
        # z*s(z) - (-z)*s(-z) = z (s(z) + s(-z)) = z
        assert abs(oracle_mod.silu(z) - oracle_mod.silu(-z) - z) < 1e-13


def test_keep_count_is_ceil_and_clamped(oracle_mod):
    assert oracle_mod.keep_count(14336, 0.3) == 4301
    assert oracle_mod.keep_count(11008, 0.3) == 3303
    assert oracle_mod.keep_count(11008, 0.1) == 1101
    assert oracle_mod.keep_count(28672, 0.3) == 8602
    assert oracle_mod.keep_count(688, 0.5) == 344
    assert oracle_mod.keep_count(4096, 0.5) == 2048
    assert oracle_mod.keep_count(100, 1.0) == 100
    assert oracle_mod.keep_count(100, 1e-9) == 1


# ------------------------------------------------------------------ a0 quantizer
def test_quantizer_recovers_exact_codes_and_power_of_two_scales(oracle_mod):
    """W = s * q with q in [-7, 7] (one +-7 per group) and s = 2^-e is exactly
    representable, so the quantizer must return q and s unchanged."""
    rng = np.random.default_rng(3)
    F, d = 24, 384
    G = d // 128
    q = rng.integers(-7, 8, size=(F, d))
    for c in range(F):
        for g in range(G):
            q[c, g * 128 + rng.integers(0, 128)] = rng.choice([-7, 7])
    e = rng.integers(3, 12, size=(F, G))
    s = np.ldexp(1.0, -e)
    w = q * np.repeat(s, 128, axis=1)
    qo, so = oracle_mod.quantize(_bf16_bits(w))
    assert np.array_equal(qo.astype(np.int64), q)
    assert np.array_equal(so, s)


def test_quantizer_invariants_on_gaussian_weights(oracle_mod):
    rng = np.random.default_rng(4)
    F, d = 40, 512
    w = _bf16_bits(rng.standard_normal((F, d)) * 0.02)
    wv = oracle_mod.bf16_bits_to_f64(w)
    q, s = oracle_mod.quantize(w)
    G = d // 128
    assert q.min() >= -8 and q.max() <= 7
    for c in range(F):
        for g in range(G):
            blk = wv[c, g * 128:(g + 1) * 128]
            qq = q[c, g * 128:(g + 1) * 128].astype(np.float64)
            amax = np.abs(blk).max()
            sc = s[c, g]
            # the stored scale is an fp16 value within half an fp16 ulp of amax/7
            assert sc == np.float16(np.float32(amax) / np.float32(7.0)).astype(np.float64)
            assert abs(sc - amax / 7) <= abs(amax / 7) * 2.0 ** -11 * 1.0001
            # reconstruction error at most half a step (plus fp32 rounding)
            assert np.all(np.abs(blk - sc * qq) <= sc * 0.5 * (1 + 1e-6) + 1e-12)
            # the largest element lands on +-7
            j = int(np.argmax(np.abs(blk)))
            assert abs(qq[j]) == 7 and np.sign(qq[j]) == np.sign(blk[j])
            assert np.all(np.abs(qq) <= 7)


def test_quantizer_zero_group(oracle_mod):
    w = np.zeros((3, 256))
    w[1, 200] = 0.5
    q, s = oracle_mod.quantize(_bf16_bits(w))
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    assert s[1, 1] == float(np.float16(np.float32(0.5) / np.float32(7)))
    assert q[1, 200] == 7 and np.count_nonzero(q) == 1


# ------------------------------------------------------------------ a1 / a3 top-k
def _brute_topk(keys, k):
    order = sorted(range(len(keys)), key=lambda j: (-keys[j], j))
    return np.array(sorted(order[:k]), dtype=np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_input_topk_matches_exhaustive_sort_with_ties(oracle_mod, seed):
    rng = np.random.default_rng(10 + seed)
    d = 128 * (1 + seed % 3)
    # few distinct magnitudes -> many exact ties; include -0.0 and +0.0
    pool = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 1.5, 3.0, -3.0, 7.25])
    x = rng.choice(pool, size=d)
    xb = _bf16_bits(x)
    mags = [abs(v) for v in oracle_mod.bf16_bits_to_f64(xb)]
    for kx in (1, d // 2, d - 3, d):
        got = oracle_mod.input_topk(xb, kx)
        assert np.array_equal(got, _brute_topk(mags, kx))


@pytest.mark.parametrize("seed", range(6))
def test_channel_topk_matches_exhaustive_sort_with_ties(oracle_mod, seed):
    rng = np.random.default_rng(20 + seed)
    F = [1, 7, 64, 333, 688, 1000][seed]
    sc = rng.integers(0, 5, size=F).astype(np.float64) * 0.25  # heavy ties
    for k in sorted({1, max(1, F // 3), F}):
        got = oracle_mod.channel_topk(sc, k)
        assert np.array_equal(got, _brute_topk(list(sc), k))
        assert len(set(got.tolist())) == k


# ------------------------------------------------------------------ a2 proxy scores
def test_proxy_one_hot_input_closed_form(oracle_mod):
    """x = v e_j: g~_c = s_gate[c][j/128] q_gate[c][j] v, u~ likewise."""
    rng = np.random.default_rng(5)
    F, d = 50, 256
    wg = _bf16_bits(rng.standard_normal((F, d)) * 0.02)
    wu = _bf16_bits(rng.standard_normal((F, d)) * 0.02)
    qg, sg = oracle_mod.quantize(wg)
    qu, su = oracle_mod.quantize(wu)
    j, v = 133, 3.5
    x = np.zeros(d)
    x[j] = v
    xb = _bf16_bits(x)
    kept = oracle_mod.input_topk(xb, d // 2)
    assert j in kept
    g, u, score = oracle_mod.proxy_scores(qg, sg, qu, su, xb, kept)
    g_ref = sg[:, j // 128] * qg[:, j] * v
    u_ref = su[:, j // 128] * qu[:, j] * v
    assert np.array_equal(g, g_ref) and np.array_equal(u, u_ref)
    want = np.abs(g_ref / (1 + np.exp(-g_ref)) * u_ref)
    assert np.allclose(score, want, rtol=1e-14, atol=0)


def test_proxy_equals_exact_state_for_quantization_exact_weights(oracle_mod):
    """With W = s*q exactly and x supported on exactly d/2 entries, the input
    keep drops only zeros and the proxy state is the exact SwiGLU state, so
    the score is |h| of Eq. (1) and the mask is the exact top-k of |h|."""
    rng = np.random.default_rng(6)
    F, d = 64, 256
    G = d // 128

    def exact_w():
        q = rng.integers(-7, 8, size=(F, d))
        for c in range(F):
            for g in range(G):
                q[c, g * 128] = 7
        return q * np.repeat(np.ldexp(1.0, -rng.integers(4, 8, size=(F, G))), 128, axis=1)

    wg, wu = exact_w(), exact_w()
    wd = rng.standard_normal((d, F)) * 0.02
    x = np.zeros(d)
    support = rng.choice(d, size=d // 2, replace=False)
    x[support] = rng.choice([-2.0, -1.0, -0.5, 0.25, 1.0, 3.0], size=d // 2)
    wgb, wub, wdb, xb = _bf16_bits(wg), _bf16_bits(wu), _bf16_bits(wd), _bf16_bits(x)
    qg, sg = oracle_mod.quantize(wgb)
    qu, su = oracle_mod.quantize(wub)
    kept = oracle_mod.input_topk(xb, d // 2)
    assert np.array_equal(np.sort(support), kept)
    g, u, score = oracle_mod.proxy_scores(qg, sg, qu, su, xb, kept)
    xv = oracle_mod.bf16_bits_to_f64(xb)
    assert np.allclose(g, oracle_mod.bf16_bits_to_f64(wgb) @ xv, rtol=1e-13, atol=1e-13)
    assert np.allclose(u, oracle_mod.bf16_bits_to_f64(wub) @ xv, rtol=1e-13, atol=1e-13)
    h, _ = oracle_mod.dense_ffn(wgb, wub, wdb, xb)
    assert np.allclose(score, np.abs(h), rtol=1e-12, atol=1e-12)


def test_proxy_uses_only_the_kept_inputs(oracle_mod):
    """Scores from x over its kept set equal scores from x~ (x zeroed outside
    the kept set) with every input kept."""
    rng = np.random.default_rng(7)
    F, d = 40, 384
    wg = _bf16_bits(rng.standard_normal((F, d)) * 0.02)
    wu = _bf16_bits(rng.standard_normal((F, d)) * 0.02)
    qg, sg = oracle_mod.quantize(wg)
    qu, su = oracle_mod.quantize(wu)
    xb = synth.bits(synth.make_x(d, 4, 20.0, seed=3))
    kept = oracle_mod.input_topk(xb, d // 2)
    xt = np.zeros(d, dtype=np.uint16)
    xt[kept] = xb[kept]
    a = oracle_mod.proxy_scores(qg, sg, qu, su, xb, kept)
    b = oracle_mod.proxy_scores(qg, sg, qu, su, xt, np.arange(d, dtype=np.int32))
    for p, r in zip(a, b):
        assert np.allclose(p, r, rtol=1e-13, atol=1e-15)
    # and x~ is not x: dropping the kept set changes the state
    c = oracle_mod.proxy_scores(qg, sg, qu, su, xb, np.arange(d, dtype=np.int32))
    assert not np.allclose(a[0], c[0])


# ------------------------------------------------------------------ Stage 2 / dense
def _tiny_layer(seed=0, F=96, d=256):
    rng = np.random.default_rng(100 + seed)
    wg = _bf16_bits(rng.standard_normal((F, d)) * 0.05)
    wu = _bf16_bits(rng.standard_normal((F, d)) * 0.05)
    wd = _bf16_bits(rng.standard_normal((d, F)) * 0.05)
    xb = synth.bits(synth.make_x(d, 2, 20.0, seed=seed))
    return wg, wu, wd, xb


def test_keep_fraction_one_equals_dense(oracle_mod):
    """Every channel selected: Stage 2 is the dense FFN of Eq. (1)."""
    wg, wu, wd, xb = _tiny_layer(1)
    r = oracle_mod.prox_ffn(wg, wu, wd, xb, 1.0)
    h, y = oracle_mod.dense_ffn(wg, wu, wd, xb)
    assert r["k"] == wg.shape[0]
    assert np.array_equal(r["idx"], np.arange(wg.shape[0]))
    assert np.allclose(r["y"], y, rtol=1e-13, atol=1e-13)
    assert np.allclose(r["h"], h, rtol=1e-13, atol=1e-13)


def test_sparse_equals_dense_with_unselected_channels_zeroed(oracle_mod):
    wg, wu, wd, xb = _tiny_layer(2)
    r = oracle_mod.prox_ffn(wg, wu, wd, xb, 0.3)
    h, _ = oracle_mod.dense_ffn(wg, wu, wd, xb)
    mask = np.zeros(wg.shape[0])
    mask[r["idx"]] = 1.0
    y_ref = oracle_mod.bf16_bits_to_f64(wd) @ (h * mask)   # library matmul
    assert np.allclose(r["y"], y_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(r["h"], h[r["idx"]], rtol=1e-13, atol=1e-13)


def test_channel_permutation_identity(oracle_mod):
    """Eq. (2): permuting channels in all three matrices leaves the FFN and,
    with the mask permuted alike, the sparse FFN unchanged."""
    wg, wu, wd, xb = _tiny_layer(3)
    F = wg.shape[0]
    perm = np.random.default_rng(9).permutation(F)
    _, y = oracle_mod.dense_ffn(wg, wu, wd, xb)
    _, yp = oracle_mod.dense_ffn(wg[perm], wu[perm], wd[:, perm], xb)
    assert np.allclose(y, yp, rtol=1e-12, atol=1e-12)
    r = oracle_mod.prox_ffn(wg, wu, wd, xb, 0.25)
    rp = oracle_mod.prox_ffn(wg[perm], wu[perm], wd[:, perm], xb, 0.25)
    inv = np.argsort(perm)
    assert np.array_equal(np.sort(perm[rp["idx"]]), r["idx"])
    assert np.allclose(r["y"], rp["y"], rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.sort(inv[r["idx"]]), rp["idx"])


def test_large_gate_reduces_to_matrix_products(oracle_mod):
    """x = e_0, W_up[:, 0] = 1 and W_gate[:, 0] = a_c: u_c = 1, g_c = a_c.
    For a_c >= 40, silu(a_c) = a_c in fp64 and y = W_down a; for a_c <= -40
    silu(a_c) ~ 0 and y ~ 0 (catches a sign flip in silu or in the gate)."""
    rng = np.random.default_rng(11)
    F, d = 32, 128
    a = rng.choice([40.0, 48.0, 64.0, 96.0], size=F)
    wg = np.zeros((F, d))
    wg[:, 0] = a
    wu = np.zeros((F, d))
    wu[:, 0] = 1.0
    wd = rng.standard_normal((d, F)) * 0.1
    x = np.zeros(d)
    x[0] = 1.0
    b = [_bf16_bits(m) for m in (wg, wu, wd, x)]
    _, y = oracle_mod.dense_ffn(*b)
    assert np.allclose(y, oracle_mod.bf16_bits_to_f64(b[2]) @ a, rtol=1e-14, atol=1e-14)
    wg[:, 0] = -a
    _, y2 = oracle_mod.dense_ffn(_bf16_bits(wg), b[1], b[2], b[3])
    assert np.max(np.abs(y2)) < 1e-12


def test_prox_composition_is_the_stage_functions_in_order(oracle_mod):
    wg, wu, wd, xb = _tiny_layer(4, F=200, d=384)
    r = oracle_mod.prox_ffn(wg, wu, wd, xb, 0.4)
    kept = oracle_mod.input_topk(xb, r["kx"])
    assert np.array_equal(kept, r["kept"])
    px = oracle_mod.Proxy(wg, wu)
    _, _, sc = oracle_mod.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    assert np.array_equal(sc, r["score"])
    idx = oracle_mod.channel_topk(sc, r["k"])
    assert np.array_equal(idx, r["idx"])
    _, y = oracle_mod.sparse_ffn(wg, wu, wd, xb, idx)
    assert np.array_equal(y, r["y"])


def test_residual_rmsnorm_closed_forms(oracle_mod):
    d = 256
    x = np.zeros(d, dtype=np.uint16)
    out = oracle_mod.residual_rmsnorm(x, np.full(d, 3.0))
    # z = 3 everywhere: 3 / sqrt(9 + 1e-6) rounds to 1.0 in bf16
    assert np.all(out == 0x3F80)
    rng = np.random.default_rng(12)
    xb = _bf16_bits(rng.standard_normal(d))
    y = rng.standard_normal(d)
    o1 = oracle_mod.bf16_bits_to_f64(oracle_mod.residual_rmsnorm(xb, y))
    rms = math.sqrt(np.mean(o1 ** 2))
    assert abs(rms - 1.0) < 5e-3
    z = oracle_mod.bf16_bits_to_f64(xb) + y
    assert np.all(np.sign(o1[np.abs(z) > 1e-3]) == np.sign(z[np.abs(z) > 1e-3]))


def _rmsnorm_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "rmsnorm_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        eps, xs, ys, want = (f.split() for f in line.split("|"))
        cases.append((float(eps[0]), [float(v) for v in xs], [float(v) for v in ys],
                      np.array([int(h, 16) for h in want], dtype=np.uint16)))
    return cases


def test_residual_rmsnorm_golden_cases(oracle_mod):
    """The stack glue against hand-worked values (tests/golden/rmsnorm_cases.txt)."""
    for eps, xs, ys, want in _rmsnorm_cases():
        got = oracle_mod.residual_rmsnorm(_bf16_bits(np.array(xs)), np.array(ys), eps)
        assert np.array_equal(got, want), (eps, xs, ys, [hex(v) for v in got])


def _bf16_rne_py(v: float) -> int:
    """bf16 bits of a double, round to nearest even (plain integer arithmetic)."""
    if v == 0.0:
        return 0
    sign = 0x8000 if v < 0 else 0
    e = math.floor(math.log2(abs(v)))
    q = abs(v) / 2.0 ** e * 128.0
    n = math.floor(q)
    if q - n > 0.5 or (q - n == 0.5 and n % 2 == 1):
        n += 1
    if n == 256:
        n, e = 128, e + 1
    return sign | ((e + 127) << 7) | (n - 128)


def test_residual_rmsnorm_golden_cases_reject_plausible_mistakes():
    """Each plausible slip in the glue (mean over d - 1, eps outside the root
    or dropped, the residual dropped, truncation instead of rounding, a
    division by the mean square) disagrees with at least one golden case, so
    the golden cases pin the definition and not just its shape."""
    def glue(xs, ys, eps, mean_div=0, eps_out=False, no_eps=False, no_res=False,
             trunc=False, no_sqrt=False):
        z = [(0.0 if no_res else a) + b for a, b in zip(xs, ys)]
        ms = sum(t * t for t in z) / (len(z) - mean_div)
        if no_eps:
            den = math.sqrt(ms)
        elif eps_out:
            den = math.sqrt(ms) + eps
        elif no_sqrt:
            den = ms + eps
        else:
            den = math.sqrt(ms + eps)
        out = []
        for t in z:
            v = t / den if den > 0 else 0.0
            if trunc:
                b = int(np.float32(v).view(np.uint32)) >> 16
            else:
                b = _bf16_rne_py(v)
            out.append(b)
        return np.array(out, dtype=np.uint16)

    cases = _rmsnorm_cases()
    # the faithful restatement reproduces every case
    for eps, xs, ys, want in cases:
        assert np.array_equal(glue(xs, ys, eps), want)
    for slip in ({"mean_div": 1}, {"eps_out": True}, {"no_eps": True}, {"no_res": True},
                 {"trunc": True}, {"no_sqrt": True}):
        assert any(not np.array_equal(glue(xs, ys, eps, **slip), want)
                   for eps, xs, ys, want in cases), slip


def _contrib_cases():
    for line in open(os.path.join(GOLDEN, "contrib_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        wd, st, k, want, idx = (f.strip() for f in line.split("|"))
        rows = [[float(v) for v in r.split()] for r in wd.split(";")]
        yield (np.array(rows), np.array([float(v) for v in st.split()]), int(k),
               np.array([float(v) for v in want.split()]), np.array([int(v) for v in idx.split()]))


def test_contrib_scores_golden_cases(oracle_mod):
    """The COUNTDOWN-style signal |h~_c| ||W_down[:, c]|| against hand-worked
    values (tests/golden/contrib_cases.txt), and the mask it keeps."""
    for wd, st, k, want, idx in _contrib_cases():
        got = oracle_mod.contrib_scores(st, _bf16_bits(wd))
        assert np.allclose(got, want, rtol=1e-15, atol=0), (got, want)
        assert np.array_equal(oracle_mod.channel_topk(got, k), idx)


def test_contrib_scores_invariants(oracle_mod):
    """Scaling one column of W_down by a power of two scales that channel's
    score by the same factor and no other; with every column of one norm the
    signal keeps the same channels as the state score; permuting the channels
    of the state scores and of W_down permutes the scores."""
    rng = np.random.default_rng(31)
    d, F = 64, 40
    wd = rng.standard_normal((d, F)) * 0.02
    st = np.abs(rng.standard_normal(F))
    base = oracle_mod.contrib_scores(st, _bf16_bits(wd))
    wd2 = oracle_mod.bf16_bits_to_f64(_bf16_bits(wd)).copy()
    wd2[:, 7] *= 4.0
    sc2 = oracle_mod.contrib_scores(st, _bf16_bits(wd2))
    assert sc2[7] == 4.0 * base[7]
    assert np.array_equal(np.delete(sc2, 7), np.delete(base, 7))
    # one column norm: a signed permutation of one column in every channel
    col = rng.standard_normal(d) * 0.02
    wd_eq = np.stack([rng.permutation(col) * rng.choice([-1.0, 1.0], size=d) for _ in range(F)], axis=1)
    sc_eq = oracle_mod.contrib_scores(st, _bf16_bits(wd_eq))
    for k in (1, 7, 20, 40):
        assert np.array_equal(oracle_mod.channel_topk(sc_eq, k), oracle_mod.channel_topk(st, k))
    perm = rng.permutation(F)
    sc_p = oracle_mod.contrib_scores(st[perm], _bf16_bits(wd)[:, perm])
    assert np.array_equal(sc_p, base[perm])


# ---------------------------------------------------------------- int8 Stage 2
def _exact_bf16_bits(v):
    """bf16 bit patterns of float values that are exact in bf16."""
    a = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert np.all(a & 0xFFFF == 0), "values must be exact in bf16"
    return (a >> 16).astype(np.uint16)


def test_q8_quantizer_invariants(oracle_mod):
    """Per-row symmetric int8: |q| <= 127; the row's largest magnitude maps to
    +-127; |w - s q| <= s/2 (plus the binary32 rounding of w/s); zero rows give q = 0,
    s = 0; each row's scale is amax / 127 of that row alone."""
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((37, 256)) * rng.uniform(0.001, 3.0, size=(37, 1))).astype(np.float32)
    w[4] = 0.0
    bits = oracle_mod.double_to_bf16(w)
    q, s = oracle_mod.quantize_rows_q8(bits)
    wf = oracle_mod.bf16_bits_to_f64(bits)
    assert np.all(np.abs(q.astype(int)) <= 127)
    assert np.all(q[4] == 0) and s[4] == 0.0
    amax = np.abs(wf).max(axis=1)
    for r in range(37):
        if r == 4:
            continue
        assert s[r] == np.float32(np.float32(amax[r]) / np.float32(127.0))
        j = int(np.argmax(np.abs(wf[r])))
        assert abs(int(q[r, j])) == 127 and np.sign(q[r, j]) == np.sign(wf[r, j])
        # w / s is rounded to binary32 before rint: |w/s| <= 127 moves it by
        # at most 127 * 2^-24, so the midpoint can be crossed by that much
        err = np.abs(wf[r] - float(s[r]) * q[r].astype(np.float64))
        assert np.all(err <= float(s[r]) * (0.5 + 127 * 2.0 ** -24))


def test_q8_quantizer_hand_worked_row(oracle_mod):
    """A row of multiples of 2^-7 whose largest magnitude is 127 * 2^-6: the
    scale is exactly 2^-6, every quotient w / s is exact, and the codes below
    are worked out by hand.  Half-way quotients go to the even integer
    (2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2), whole ones stay."""
    u = 2.0 ** -6
    row = np.array([127, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -127, 0, 64, -0.5, 126.5]) * u
    want = np.array([127, 2, 4, -2, -4, 0, 2, -127, 0, 64, 0, 126], dtype=np.int8)
    bits = oracle_mod.double_to_bf16(row.reshape(1, -1))
    assert np.array_equal(oracle_mod.bf16_bits_to_f64(bits).ravel(), row)  # exact in bf16
    q, s = oracle_mod.quantize_rows_q8(bits)
    assert s[0] == np.float32(u)
    assert np.array_equal(q[0], want)


def test_q8_stage2_reduces_to_bf16_stage2_on_exact_weights(oracle_mod):
    """Weights w = 2^-6 q_true with integer |q_true| <= 127 and every row (and
    W_down column) reaching 127 are exact in bf16 and quantize exactly (s =
    2^-6), so the int8 Stage 2 equals the bf16 Stage 2 (an independent
    function of the oracle) on any channel set."""
    rng = np.random.default_rng(6)
    F, d = 96, 128
    def exact(rows, cols, col_major=False):
        qt = rng.integers(-127, 128, size=(rows, cols))
        if col_major:
            qt[rng.integers(0, rows, size=cols), np.arange(cols)] = 127
        else:
            qt[np.arange(rows), rng.integers(0, cols, size=rows)] = -127
        return qt, _exact_bf16_bits(qt.astype(np.float32) * np.float32(2.0 ** -6))
    qg_t, wg = exact(F, d)
    qu_t, wu = exact(F, d)
    qd_t, wd = exact(d, F, col_major=True)   # W_down [d][F]: each column reaches 127
    x = synth.bits(synth.make_x(d, 3, 20.0, 9))
    q8 = oracle_mod.stage2_q8(wg, wu, wd)
    assert np.array_equal(q8["q_gate"], qg_t) and np.array_equal(q8["q_up"], qu_t)
    assert np.array_equal(q8["q_down"], qd_t.T)
    assert np.all(q8["s_gate"] == np.float32(2.0 ** -6)) and np.all(q8["s_down"] == np.float32(2.0 ** -6))
    idx = np.sort(rng.choice(F, size=40, replace=False)).astype(np.int32)
    h8, y8 = oracle_mod.sparse_ffn_q8(q8, x, idx)
    h, y = oracle_mod.sparse_ffn(wg, wu, wd, x, idx)
    assert np.allclose(h8, h, rtol=1e-12, atol=1e-12 * np.abs(h).max())
    assert np.allclose(y8, y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_q8_stage2_one_channel_closed_form(oracle_mod):
    """One selected channel: y = silu(s_g q_g.x) (s_u q_u.x) s_d q_d, written
    out for a tiny case with hand-set codes."""
    d, F = 128, 2
    q8 = {"q_gate": np.zeros((F, d), np.int8), "s_gate": np.array([0.5, 1.0], np.float32),
          "q_up": np.zeros((F, d), np.int8), "s_up": np.array([0.25, 1.0], np.float32),
          "q_down": np.zeros((F, d), np.int8), "s_down": np.array([2.0, 1.0], np.float32)}
    q8["q_gate"][0, 3] = 4      # g = 0.5 * 4 * x3
    q8["q_up"][0, 5] = -8       # u = 0.25 * -8 * x5
    q8["q_down"][0, 7] = 3      # y7 = h * 2 * 3
    q8["q_down"][1, 7] = 100    # channel 1 is not selected
    xs = np.zeros(d, np.float32)
    xs[3], xs[5] = 1.5, -2.0
    x = _exact_bf16_bits(xs)
    h, y = oracle_mod.sparse_ffn_q8(q8, x, np.array([0], np.int32))
    g, u = 0.5 * 4 * 1.5, 0.25 * -8 * -2.0
    hh = g / (1 + np.exp(-g)) * u
    assert np.isclose(h[0], hh, rtol=1e-15)
    expect = np.zeros(d)
    expect[7] = hh * 2.0 * 3
    assert np.allclose(y, expect, rtol=1e-15, atol=0)


# ------------------------------------------------------ block-granular mask
def test_block_topk_golden_cases(oracle_mod):
    """Hand-worked cases of the block mask (PrunePath Sec. 2.2 Eq. (2) blocks;
    expert score = sum of its channels' scores, ties to the lower expert)."""
    n = 0
    for line in open(os.path.join(GOLDEN, "block_topk_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        bw, K, sc, want = [f.strip() for f in line.split("|")]
        sc = np.array([float(v) for v in sc.split()])
        want = np.array([int(v) for v in want.split()], dtype=np.int32)
        idx, S = oracle_mod.block_topk(sc, int(bw), int(K))
        assert np.array_equal(idx, want), (line, idx)
        assert S.size == sc.size // int(bw)
        n += 1
    assert n >= 8


def test_block_topk_width_one_is_the_channel_topk(oracle_mod):
    rng = np.random.default_rng(7)
    sc = np.round(rng.exponential(size=500), 2)  # many exact ties
    for k in (1, 17, 250, 500):
        idx, _ = oracle_mod.block_topk(sc, 1, k)
        assert np.array_equal(idx, oracle_mod.channel_topk(sc, k))


def test_block_topk_keeps_whole_blocks_and_agrees_with_block_constant_channel_topk(oracle_mod):
    """With every channel of a block carrying the same value v_e, the block
    mask equals the channel top-(K bw): a channel ranking whose ties go to
    the lower channel takes blocks whole, in order of v_e."""
    rng = np.random.default_rng(8)
    for bw, E in ((4, 64), (16, 37), (64, 20)):
        v = rng.permutation(E).astype(np.float64) + 1.0  # distinct
        sc = np.repeat(v, bw)
        for K in (1, E // 3, E):
            idx, S = oracle_mod.block_topk(sc, bw, K)
            assert np.array_equal(S, v * bw)
            assert idx.size == K * bw
            assert np.array_equal(idx, oracle_mod.channel_topk(sc, K * bw))
            blocks = idx.reshape(K, bw)
            assert np.all(blocks == blocks[:, :1] + np.arange(bw))  # whole, contiguous


def test_block_topk_follows_a_permutation_of_the_blocks(oracle_mod):
    """Eq. (2) is stated for any permutation: relabelling the experts relabels
    the kept set (distinct expert sums, so no tie decides)."""
    rng = np.random.default_rng(9)
    bw, E, K = 8, 50, 13
    sc = rng.random(bw * E)
    perm = rng.permutation(E)
    sc_p = sc.reshape(E, bw)[perm].ravel()  # expert e of sc_p is expert perm[e] of sc
    idx, _ = oracle_mod.block_topk(sc, bw, K)
    idx_p, _ = oracle_mod.block_topk(sc_p, bw, K)
    kept = set(idx.reshape(K, bw)[:, 0] // bw)
    kept_p = set(idx_p.reshape(K, bw)[:, 0] // bw)
    assert kept == {int(perm[e]) for e in kept_p}


def test_block_topk_rejects_ragged_widths(oracle_mod):
    with pytest.raises(Exception):
        oracle_mod.block_topk(np.ones(10), 4, 1)  # 10 channels do not split into blocks of 4
    with pytest.raises(Exception):
        oracle_mod.block_topk(np.ones(8), 2, 5)   # only 4 blocks


def test_q4_quantizer_invariants(oracle_mod):
    """Per-row symmetric int4: -8 <= q <= 7 (|q| <= 7 from a symmetric scale);
    the row's largest magnitude maps to +-7; |w - s q| <= s/2 (plus the
    binary32 rounding of w/s); zero rows give q = 0, s = 0; each row's scale is
    amax / 7 of that row alone."""
    rng = np.random.default_rng(15)
    w = (rng.standard_normal((29, 256)) * rng.uniform(0.001, 3.0, size=(29, 1))).astype(np.float32)
    w[6] = 0.0
    bits = oracle_mod.double_to_bf16(w)
    q, s = oracle_mod.quantize_rows_q4(bits)
    wf = oracle_mod.bf16_bits_to_f64(bits)
    assert np.all(q >= -7) and np.all(q <= 7)
    assert np.all(q[6] == 0) and s[6] == 0.0
    amax = np.abs(wf).max(axis=1)
    for r in range(29):
        if r == 6:
            continue
        assert s[r] == np.float32(np.float32(amax[r]) / np.float32(7.0))
        j = int(np.argmax(np.abs(wf[r])))
        assert abs(int(q[r, j])) == 7 and np.sign(q[r, j]) == np.sign(wf[r, j])
        err = np.abs(wf[r] - float(s[r]) * q[r].astype(np.float64))
        assert np.all(err <= float(s[r]) * (0.5 + 7 * 2.0 ** -24))


def test_q4_quantizer_hand_worked_row(oracle_mod):
    """A row whose largest magnitude is 7 * 2^-3: the scale is exactly 2^-3,
    every quotient w / s is exact, and the codes are worked out by hand.
    Half-way quotients go to the even integer (2.5 -> 2, 3.5 -> 4, -0.5 -> 0,
    6.5 -> 6, -5.5 -> -6), whole ones stay."""
    u = 2.0 ** -3
    row = np.array([7, 2.5, 3.5, -0.5, 6.5, -5.5, -7, 0, 1, -3]) * u
    want = np.array([7, 2, 4, 0, 6, -6, -7, 0, 1, -3], dtype=np.int8)
    bits = oracle_mod.double_to_bf16(row.reshape(1, -1))
    assert np.array_equal(oracle_mod.bf16_bits_to_f64(bits).ravel(), row)  # exact in bf16
    q, s = oracle_mod.quantize_rows_q4(bits)
    assert s[0] == np.float32(u)
    assert np.array_equal(q[0], want)


def test_q4_stage2_reduces_to_bf16_stage2_on_exact_weights(oracle_mod):
    """Weights w = 2^-3 q_true with integer |q_true| <= 7 and every row (and
    W_down column) reaching 7 are exact in bf16 and quantize exactly (s =
    2^-3), so the int4 Stage 2 equals the bf16 Stage 2 (an independent
    function of the oracle) on any channel set."""
    rng = np.random.default_rng(16)
    F, d = 80, 128
    def exact(rows, cols, col_major=False):
        qt = rng.integers(-7, 8, size=(rows, cols))
        if col_major:
            qt[rng.integers(0, rows, size=cols), np.arange(cols)] = 7
        else:
            qt[np.arange(rows), rng.integers(0, cols, size=rows)] = -7
        return qt, _exact_bf16_bits(qt.astype(np.float32) * np.float32(2.0 ** -3))
    qg_t, wg = exact(F, d)
    qu_t, wu = exact(F, d)
    qd_t, wd = exact(d, F, col_major=True)
    x = synth.bits(synth.make_x(d, 3, 20.0, 19))
    q4 = oracle_mod.stage2_q4(wg, wu, wd)
    assert np.array_equal(q4["q_gate"], qg_t) and np.array_equal(q4["q_up"], qu_t)
    assert np.array_equal(q4["q_down"], qd_t.T)
    assert np.all(q4["s_gate"] == np.float32(2.0 ** -3)) and np.all(q4["s_down"] == np.float32(2.0 ** -3))
    idx = np.sort(rng.choice(F, 23, replace=False)).astype(np.int32)
    h4, y4 = oracle_mod.sparse_ffn_q8(q4, x, idx)
    h, y = oracle_mod.sparse_ffn(wg, wu, wd, x, idx)
    assert np.allclose(h4, h, rtol=1e-12, atol=1e-12)
    assert np.allclose(y4, y, rtol=1e-12, atol=1e-12 * max(1.0, np.abs(y).max()))
