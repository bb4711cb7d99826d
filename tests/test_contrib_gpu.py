"""The second selection signal on the GPU vs the oracle, through the C ABI
(marked gpu).

prox_ffn_contrib ranks channel c by |silu(g~_c) u~_c| * ||W_down[:, c]||_2:
the magnitude of channel c's term in the down projection's linear
combination y = sum_c h_c W_down[:, c] ("COUNTDOWN", Abstract), with the
Prox proxy state as the coefficient.  Bars as for prox_ffn: every score
within half the tie band of the oracle's, the mask exact outside the tie
band around the oracle's k-th score, y within max-abs 2e-2 and relative-L2
1e-2 (and 1e-3 of max |y|) of the oracle's Stage 2 on the GPU's mask.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import ATOL_Y, RTOL_L2_Y, TIE_BAND, host_bits, tie_band_mask_check, y_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _check_contrib(prox, L, w, x, rho, px=None):
    wg, wu, wd = w
    xb = host_bits(x)
    r = prox.prox_ffn_contrib_debug(L, x.cuda(), rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    k = oracle.keep_count(L.d_ff, rho)
    assert r["k"] == k
    kept = oracle.input_topk(xb, oracle.keep_count(L.d_model, 0.5))
    if px is None:
        px = oracle.Proxy(wg, wu)
    _, _, state = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    sc = oracle.contrib_scores(state, wd)
    sc_gpu = r["scores"].cpu().numpy().astype(np.float64)
    kth = np.sort(sc)[::-1][k - 1]
    scale = max(kth, float(np.median(sc)), 1e-30)
    rel = np.abs(sc_gpu - sc) / np.maximum(np.abs(sc), scale)
    assert rel.max() < TIE_BAND / 2, rel.max()
    idx = r["idx"].cpu().numpy()
    bad, in_band = tie_band_mask_check(idx, sc, k)
    assert bad == 0, f"{bad} channels outside the tie band disagree ({in_band} in band)"
    h_or, y_or = oracle.sparse_ffn(wg, wu, wd, xb, idx)
    mx, rl = y_errors(r["y"].cpu().numpy(), y_or)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max())
    hh = r["h"].cpu().numpy().astype(np.float64)
    assert np.allclose(hh, h_or, rtol=1e-4, atol=1e-4 * np.abs(h_or).max())
    # the plain entry point selects the same channels: only the order of the
    # output additions differs
    y = prox.prox_ffn_contrib(L, x.cuda(), rho)
    torch.cuda.synchronize()
    assert torch.allclose(y, r["y"], rtol=0, atol=1e-5 * float(r["y"].abs().max()))
    return r, state, sc


def _layer(prox, d, F, seed, col_scale=None):
    wg, wu, wd = synth.make_weights(d, F, 0.02, seed)
    if col_scale is not None:  # columns of W_down with different norms
        wd = (wd.float() * col_scale[None, :]).to(torch.bfloat16)
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    return L, (host_bits(wg), host_bits(wu), host_bits(wd))


@pytest.mark.parametrize("d,F,rho", [(256, 688, 0.5), (1024, 3000, 0.3), (512, 3000, 0.1),
                                     (2048, 5000, 0.3)])
def test_contrib_matches_oracle(prox, d, F, rho):
    cs = torch.exp(torch.randn(F, generator=torch.Generator().manual_seed(F)) * 0.5)
    L, w = _layer(prox, d, F, seed=3 * d + F, col_scale=cs)
    for s in range(2):
        _check_contrib(prox, L, w, synth.make_x(d, max(1, d // 100), 20.0, 300 + s), rho)


def test_contrib_signal_changes_the_mask(prox):
    """With W_down columns of different norms the contribution signal keeps a
    different set of channels than the state signal (prox_ffn), and each
    matches its own oracle."""
    d, F, rho = 1024, 3000, 0.3
    cs = torch.exp(torch.randn(F, generator=torch.Generator().manual_seed(5)) * 0.7)
    L, w = _layer(prox, d, F, seed=77, col_scale=cs)
    x = synth.make_x(d, 10, 20.0, 78)
    r, state, sc = _check_contrib(prox, L, w, x, rho)
    k = oracle.keep_count(F, rho)
    m_state = set(oracle.channel_topk(state, k).tolist())
    m_contrib = set(r["idx"].cpu().numpy().tolist())
    assert len(m_state ^ m_contrib) > k // 10


def test_contrib_full_size_layer(prox):
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    px = oracle.Proxy.__new__(oracle.Proxy)
    px.q_gate, px.s_gate = oracle.quantize(w[0])
    px.q_up, px.s_up = oracle.quantize(w[1])
    _check_contrib(prox, L, w, synth.hidden(shape, seed=1), 0.3, px=px)
