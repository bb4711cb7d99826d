"""Helpers shared by the parity tests: decode the documented device layouts
(include/prox.h) on the host and compare results with the oracle."""
import numpy as np
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth

ATOL_Y = 2e-2      # max-abs error bound on y
RTOL_L2_Y = 1e-2   # relative L2 error bound on y
TIE_BAND = 1e-4    # channels within this relative distance of the k-th score may differ


def padded_ff(F):
    return (F + 63) // 64 * 64


def decode_proxy(layer):
    """(q_gate[F][d], q_up[F][d], s_gate[F][G], s_up[F][G]) from the device buffers."""
    d, F = layer.d_model, layer.d_ff
    Fp, G = padded_ff(F), d // 128
    P = layer.bufs["proxy_codes"].cpu().numpy()[: d * Fp].reshape(d, Fp)
    qg = ((P & 0x0F).astype(np.int16) - 8).astype(np.int8)[:, :F].T.copy()
    qu = ((P >> 4).astype(np.int16) - 8).astype(np.int8)[:, :F].T.copy()
    S = layer.bufs["proxy_scales"].cpu().numpy()[: G * Fp * 4].view(np.float16).reshape(G, Fp, 2)
    sg = S[:, :F, 0].T.astype(np.float64)
    su = S[:, :F, 1].T.astype(np.float64)
    pad = P[:, F:]
    return qg, qu, sg, su, pad, S[:, F:, :]


def host_bits(t):
    return synth.bits(t)


def tie_band_mask_check(idx_gpu, score_oracle, k, band=TIE_BAND):
    """The GPU mask must hold exactly k distinct channels and agree with the
    oracle's top-k on every channel whose oracle score lies outside the tie
    band around the oracle's k-th score.  Returns (n_disagree_outside, n_in_band)."""
    idx_gpu = np.asarray(idx_gpu)
    F = score_oracle.size
    assert idx_gpu.size == k
    assert np.unique(idx_gpu).size == k
    assert idx_gpu.min() >= 0 and idx_gpu.max() < F
    assert np.all(np.diff(idx_gpu) > 0), "channel list must be ascending"
    sel_gpu = np.zeros(F, bool)
    sel_gpu[idx_gpu] = True
    idx_or = oracle.channel_topk(score_oracle, k)
    sel_or = np.zeros(F, bool)
    sel_or[idx_or] = True
    kth = np.sort(score_oracle)[::-1][k - 1]
    band_mask = np.abs(score_oracle - kth) <= band * abs(kth)
    outside = ~band_mask
    return int(np.count_nonzero(sel_gpu[outside] != sel_or[outside])), int(band_mask.sum())


def y_errors(y_gpu, y_ref):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    rel = np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-30)
    return float(err.max()), float(rel)


def check_step(prox, L, w, x, rho, kappa=0.5, px=None):
    """One decode step through prox_ffn_debug against the oracle: the kept
    inputs bit-exact, every score within half the tie band, the mask exact
    outside the band, y and h within the bars on the GPU's own mask.  Returns
    the debug outputs."""
    wg, wu, wd = w
    xb = host_bits(x)
    r = prox.prox_ffn_debug(L, x.cuda(), rho, kappa)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    kx, k = oracle.keep_count(L.d_model, kappa), oracle.keep_count(L.d_ff, rho)
    assert (r["kx"], r["k"]) == (kx, k)
    # input sparsity: bit-exact
    kept_or = oracle.input_topk(xb, kx)
    assert np.array_equal(r["kept"].cpu().numpy(), kept_or)
    # proxy scores and the mask
    if px is None:
        px = oracle.Proxy(wg, wu)
    g, u, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept_or)
    sc_gpu = r["scores"].cpu().numpy().astype(np.float64)
    # fp32 proxy vs fp64 oracle, measured on the ranking scale: the k-th score
    # (or the median score, when k is so large that the k-th is near zero).
    # The bound is half the tie band: with every score within band/2 of the
    # oracle's, no two channels whose oracle scores lie outside the band around
    # the k-th can change order, so the band covers all fp32 rounding.  (An fp32
    # sum of k_x products that cancel to ~1/sqrt(k_x) of their magnitude sum
    # carries ~sqrt(k_x) * 2^-24 relative error: about 1e-5 at k_x = 4096.)
    kth = np.sort(sc)[::-1][k - 1]
    scale = max(kth, float(np.median(sc)), 1e-30)
    rel = np.abs(sc_gpu - sc) / np.maximum(np.abs(sc), scale)
    assert rel.max() < TIE_BAND / 2, rel.max()
    idx = r["idx"].cpu().numpy()
    bad, in_band = tie_band_mask_check(idx, sc, k)
    assert bad == 0, f"{bad} channels outside the tie band disagree ({in_band} in band)"
    # Stage 2 on the GPU's mask
    h_or, y_or = oracle.sparse_ffn(wg, wu, wd, xb, idx)
    mx, rl = y_errors(r["y"].cpu().numpy(), y_or)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max())  # fp32 path: far inside the bar
    hh = r["h"].cpu().numpy().astype(np.float64)
    assert np.allclose(hh, h_or, rtol=1e-4, atol=1e-4 * np.abs(h_or).max())
    return r
