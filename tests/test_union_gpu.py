"""A batch over the union of its tokens' masks (prox_ffn_batch_union) vs the
oracle, through the C ABI (marked gpu).

Every token keeps its own exact mask and output (Prox, Abstract: one mask
per token from its proxy ranking); only the Stage-2 reads are shared.  Per
token: the mask exact outside the tie band around the oracle's k-th score,
and the same channels that prox_ffn selects for that token alone; y_t within
max-abs 2e-2 and relative-L2 1e-2 (and 1e-3 of max |y|) of the oracle's
sparse FFN on that mask, and equal to prox_ffn's y_t up to the order of the
fp32 additions.  Batches larger than one pass run in several passes.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import ATOL_Y, RTOL_L2_Y, host_bits, tie_band_mask_check, y_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _layer(prox, d, F, seed):
    wg, wu, wd = synth.make_weights(d, F, 0.02, seed)
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    return L, (host_bits(wg), host_bits(wu), host_bits(wd))


def _tokens(d, B, seed):
    return torch.stack([synth.make_x(d, max(1, d // 100), 20.0, seed + t) for t in range(B)])


def _check_batch(prox, L, w, X, rho, px=None):
    """Union batch vs the oracle and vs single-token steps, token by token."""
    B, d = X.shape
    r = prox.prox_ffn_batch_union_debug(L, X.cuda(), rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    k = oracle.keep_count(L.d_ff, rho)
    if px is None:
        px = oracle.Proxy(w[0], w[1])
    union = np.zeros(L.d_ff, bool)
    for t in range(B):
        xb = host_bits(X[t])
        mask = r["masks"][t].cpu().numpy()
        union[mask] = True
        kept = oracle.input_topk(xb, oracle.keep_count(d, 0.5))
        _, _, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
        bad, in_band = tie_band_mask_check(mask, sc, k)
        assert bad == 0, (t, bad, in_band)
        _, y_or = oracle.sparse_ffn(*w, xb, mask)
        yt = r["y"][t].cpu().numpy()
        mx, rl = y_errors(yt, y_or)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (t, mx, rl)
        assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()), (t, mx)
        # the same mask and output as the token's own step
        one = prox.prox_ffn_debug(L, X[t].cuda(), rho)
        torch.cuda.synchronize()
        assert np.array_equal(one["idx"].cpu().numpy(), mask), t
        scale = float(one["y"].abs().max())
        assert torch.allclose(r["y"][t], one["y"], rtol=0, atol=1e-5 * max(scale, 1e-30)), t
    # no channel outside every mask carries a bit
    m = r["member"].cpu().numpy()
    assert np.array_equal(m != 0, union)
    assert np.all(m < (1 << B))
    return r


@pytest.mark.parametrize("d,F,B,rho", [(256, 688, 1, 0.3), (256, 688, 8, 0.5), (1024, 3000, 8, 0.3),
                                       (512, 3000, 5, 0.1), (2048, 5000, 8, 0.3)])
def test_union_batch_matches_oracle(prox, d, F, B, rho):
    L, w = _layer(prox, d, F, seed=7 * d + F)
    assert prox.prox_batch_union_group(L) >= B
    _check_batch(prox, L, w, _tokens(d, B, 500 + B), rho)


def test_union_batch_in_several_passes(prox):
    """19 tokens: passes of G, G and the rest; every token as in its own step."""
    d, F, rho = 1024, 3000, 0.3
    L, w = _layer(prox, d, F, seed=99)
    G = prox.prox_batch_union_group(L)
    B = 2 * G + 3
    X = _tokens(d, B, 900)
    y = prox.prox_ffn_batch_union(L, X.cuda(), rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    for t in range(B):
        one = prox.prox_ffn(L, X[t].cuda(), rho)
        torch.cuda.synchronize()
        scale = float(one.abs().max())
        assert torch.allclose(y[t], one, rtol=0, atol=1e-5 * scale), t
    # and against the oracle for the tokens of the last pass
    _check_batch(prox, L, w, X[2 * G:], rho)


def test_union_batch_identical_tokens(prox):
    """Eight copies of one token: one mask, every row read once, eight outputs
    equal up to the order of the fp32 additions (y is accumulated with
    atomic adds from several CTAs)."""
    d, F = 1024, 3000
    L, w = _layer(prox, d, F, seed=5)
    X = _tokens(d, 1, 77).repeat(8, 1)
    r = _check_batch(prox, L, w, X, 0.3)
    m = r["member"].cpu().numpy()
    assert set(np.unique(m).tolist()) <= {0, 255}
    scale = float(r["y"][0].abs().max())
    for t in range(1, 8):
        assert torch.allclose(r["y"][t], r["y"][0], rtol=0, atol=1e-5 * scale)


def test_union_batch_full_size_layer(prox):
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    px = oracle.Proxy.__new__(oracle.Proxy)
    px.q_gate, px.s_gate = oracle.quantize(w[0])
    px.q_up, px.s_up = oracle.quantize(w[1])
    G = prox.prox_batch_union_group(L)
    assert G == 8
    X = torch.stack([synth.hidden(shape, seed=10 + t) for t in range(G)])
    _check_batch(prox, L, w, X, 0.3, px=px)


def test_union_batch_argument_errors(prox):
    d, F = 256, 688
    L, _ = _layer(prox, d, F, seed=3)
    X = _tokens(d, 4, 1).cuda()
    y = torch.empty(4, d, dtype=torch.float32, device="cuda")
    lib = prox._load()
    assert lib.prox_ffn_batch_union(L.handle, X.data_ptr(), 0, 0.3, y.data_ptr(), None) == \
        prox.PROX_ERR_INVALID_ARG
    assert lib.prox_ffn_batch_union(L.handle, X.data_ptr(), 4, 1.5, y.data_ptr(), None) == \
        prox.PROX_ERR_INVALID_ARG
    # x inside y
    assert lib.prox_ffn_batch_union(L.handle, y.data_ptr(), 4, 0.3, y.data_ptr(), None) == \
        prox.PROX_ERR_INVALID_ARG
    G = prox.prox_batch_union_group(L)
    Xb = _tokens(d, G + 1, 2).cuda()
    yb = torch.empty(G + 1, d, dtype=torch.float32, device="cuda")
    mem = torch.zeros(F, dtype=torch.int32, device="cuda")
    assert lib.prox_ffn_batch_union_debug(L.handle, Xb.data_ptr(), G + 1, 0.3, yb.data_ptr(),
                                          mem.data_ptr(), None) == prox.PROX_ERR_INVALID_ARG
    # int8 Stage-2 rows are not supported by the union pass
    wg, wu, wd = synth.make_weights(d, F, 0.02, 4, device="cuda")
    Lq = prox.prox_prepare_q8(wg, wu, wd)
    assert prox.prox_batch_union_group(Lq) == 0
    assert lib.prox_ffn_batch_union(Lq.handle, X.data_ptr(), 4, 0.3, y.data_ptr(), None) == \
        prox.PROX_ERR_UNSUPPORTED_SHAPE
    assert prox.prox_get_status(L) == 0


def test_union_batch_grouped_stage1_llama2_7b(prox):
    """Five tokens of a Llama-2-7B layer: Stage 1 of all five runs in one
    launch (a group of CTAs per token, chunks wider than a CTA's threads);
    each token's mask and y as in its own step and against the oracle."""
    shape = synth.LLAMA2_7B
    wg, wu, wd = synth.layer(shape, seed=3, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    px = oracle.Proxy.__new__(oracle.Proxy)
    px.q_gate, px.s_gate = oracle.quantize(w[0])
    px.q_up, px.s_up = oracle.quantize(w[1])
    X = torch.stack([synth.hidden(shape, seed=40 + t) for t in range(5)])
    for rho in (0.3, 0.1):
        _check_batch(prox, L, w, X, rho, px=px)


def test_union_batch_with_all_tied_tokens(prox):
    """Zero tokens among ordinary ones, on the Llama-3-8B layer (grouped
    Stage 1): a zero token's scores all tie, so its mask is the first k
    channels and its y is 0; the other tokens are unaffected."""
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    del wg, wu, wd
    X = torch.stack([synth.hidden(shape, seed=60 + t) for t in range(6)])
    X[1].zero_()
    X[4].zero_()
    r = prox.prox_ffn_batch_union_debug(L, X.cuda(), 0.3)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    k = oracle.keep_count(shape.d_ff, 0.3)
    for t in (1, 4):
        assert np.array_equal(r["masks"][t].cpu().numpy(), np.arange(k))
        assert torch.count_nonzero(r["y"][t]) == 0
    for t in (0, 2, 3, 5):
        one = prox.prox_ffn_debug(L, X[t].cuda(), 0.3)
        torch.cuda.synchronize()
        assert np.array_equal(one["idx"].cpu().numpy(), r["masks"][t].cpu().numpy()), t
        scale = float(one["y"].abs().max())
        assert torch.allclose(r["y"][t], one["y"], rtol=0, atol=1e-5 * scale), t


def test_union_batch_llama3_70b_layer(prox):
    """Seven tokens of a Llama-3-70B layer: the proxy needs 28 CTAs per token,
    so Stage 1 runs as a launch of 5 token groups and one of 2.  Every
    token's mask equals its own step's and y_t matches it and the oracle's
    sparse FFN on that mask."""
    shape = synth.LLAMA3_70B
    wg, wu, wd = synth.layer(shape, seed=1, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    G = prox.prox_batch_union_group(L)
    assert G >= 5
    X = torch.stack([synth.hidden(shape, seed=80 + t) for t in range(G)])
    r = prox.prox_ffn_batch_union_debug(L, X.cuda(), 0.3)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    k = oracle.keep_count(shape.d_ff, 0.3)
    for t in range(G):
        mask = r["masks"][t].cpu().numpy()
        assert mask.size == k
        one = prox.prox_ffn_debug(L, X[t].cuda(), 0.3)
        torch.cuda.synchronize()
        assert np.array_equal(one["idx"].cpu().numpy(), mask), t
        scale = float(one["y"].abs().max())
        assert torch.allclose(r["y"][t], one["y"], rtol=0, atol=1e-5 * scale), t
        _, y_or = oracle.sparse_ffn(*w, host_bits(X[t]), mask)
        mx, rl = y_errors(r["y"][t].cpu().numpy(), y_or)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (t, mx, rl)
