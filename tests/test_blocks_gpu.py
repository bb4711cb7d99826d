"""Block-granular masks on the GPU vs the oracle, through the C ABI (marked gpu).

prox_ffn_blocks keeps the K = ceil(rho E) experts of block_width contiguous
channels whose summed proxy score is largest ("PrunePath", Sec. 2.2 Eq. (2)
experts; Sec. 3.1 activates a subset; the weights are taken as already
permuted).  Bars: per-channel scores as in the channel-mask tests; the mask
is whole, aligned blocks, K of them, equal to the oracle's block top-K on
every block whose oracle sum lies outside the tie band (1e-4 relative to the
K-th sum); y within max-abs 2e-2 and relative-L2 1e-2 (and 1e-3 of max |y|)
of the oracle's Stage 2 on the GPU's mask.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import ATOL_Y, RTOL_L2_Y, TIE_BAND, host_bits, y_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _layer(prox, d, F, seed, sigma=0.02):
    wg, wu, wd = synth.make_weights(d, F, sigma, seed)
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    return L, (host_bits(wg), host_bits(wu), host_bits(wd))


def _check_blocks(prox, L, w, x, bw, rho, px=None):
    wg, wu, wd = w
    xb = host_bits(x)
    r = prox.prox_ffn_blocks_debug(L, x.cuda(), bw, rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    F = L.d_ff
    E = F // bw
    K = oracle.keep_count(E, rho)
    assert r["k"] == K * bw
    kept = oracle.input_topk(xb, oracle.keep_count(L.d_model, 0.5))
    if px is None:
        px = oracle.Proxy(wg, wu)
    _, _, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    sc_gpu = r["scores"].cpu().numpy().astype(np.float64)
    scale = max(float(np.median(sc)), 1e-30)
    assert (np.abs(sc_gpu - sc) / np.maximum(np.abs(sc), scale)).max() < TIE_BAND / 2
    # whole, aligned, ascending blocks
    idx = r["idx"].cpu().numpy()
    assert idx.size == K * bw and np.all(np.diff(idx) > 0)
    blk = idx.reshape(K, bw)
    assert np.all(blk[:, 0] % bw == 0) and np.all(blk == blk[:, :1] + np.arange(bw))
    got = set((blk[:, 0] // bw).tolist())
    # the oracle's block top-K, exact outside the tie band
    idx_or, S = oracle.block_topk(sc, bw, K)
    want = set((idx_or.reshape(K, bw)[:, 0] // bw).tolist())
    SK = np.sort(S)[::-1][K - 1]
    band = np.abs(S - SK) <= TIE_BAND * abs(SK)
    for e in range(E):
        if not band[e]:
            assert (e in got) == (e in want), (e, S[e], SK)
    # Stage 2 on the GPU's mask
    h_or, y_or = oracle.sparse_ffn(wg, wu, wd, xb, idx)
    mx, rl = y_errors(r["y"].cpu().numpy(), y_or)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()), mx
    hh = r["h"].cpu().numpy().astype(np.float64)
    assert np.allclose(hh, h_or, rtol=1e-4, atol=1e-4 * np.abs(h_or).max())
    # the plain entry point: the same mask, so only the order of the output additions differs
    y = prox.prox_ffn_blocks(L, x.cuda(), bw, rho)
    torch.cuda.synchronize()
    assert torch.allclose(y, r["y"], rtol=1e-5, atol=1e-6 * float(np.abs(y_or).max()))
    return r


@pytest.mark.parametrize("d,F,bw,rho", [(256, 688, 4, 0.5), (1024, 4736, 32, 0.3),
                                        (512, 9472, 64, 0.3), (2048, 5000, 8, 0.1),
                                        (128, 19200, 128, 0.5)])
def test_block_mask_matches_oracle(prox, d, F, bw, rho):
    L, w = _layer(prox, d, F, seed=3 * d + F + bw)
    if F // bw < prox.prox_layer_blocks(L):
        pytest.skip("fewer blocks than CTAs on this device")
    for s in range(2):
        _check_blocks(prox, L, w, synth.make_x(d, max(1, d // 100), 20.0, 70 + s), bw, rho)


def test_block_mask_extremes(prox):
    d, F = 256, 688
    L, w = _layer(prox, d, F, seed=5)
    x = synth.make_x(d, 4, 20.0, 6)
    r = _check_blocks(prox, L, w, x, 4, 1.0)  # every block: the dense FFN
    y_dense = prox.prox_dense_ffn(L, x.cuda())
    torch.cuda.synchronize()
    assert torch.allclose(r["y"], y_dense, rtol=1e-5, atol=1e-5)
    _check_blocks(prox, L, w, x, 4, 1e-6)  # one block


def test_block_widths_are_checked(prox):
    d, F = 256, 688
    L, _ = _layer(prox, d, F, seed=7)
    x = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    for bw, code in ((3, prox.PROX_ERR_INVALID_ARG), (0, prox.PROX_ERR_INVALID_ARG),
                     (512, prox.PROX_ERR_INVALID_ARG), (32, prox.PROX_ERR_UNSUPPORTED_SHAPE),
                     (8, prox.PROX_ERR_UNSUPPORTED_SHAPE)):
        with pytest.raises(prox.ProxError) as e:  # 688 / 32 is not whole; 688 / 8 = 86 < CTAs
            prox.prox_ffn_blocks(L, x, bw, 0.3)
        assert e.value.code == code, bw


def test_block_mask_is_deterministic_and_full_size(prox):
    """The Llama-3-8B-shaped layer at keep fraction 0.3 with 64-channel blocks
    (the measured block workload), twice with the same mask."""
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    px = oracle.Proxy(w[0], w[1])
    x = synth.hidden(shape, seed=1)
    r1 = _check_blocks(prox, L, w, x, 64, 0.3, px=px)
    r2 = prox.prox_ffn_blocks_debug(L, x.cuda(), 64, 0.3)
    torch.cuda.synchronize()
    assert torch.equal(r1["idx"], r2["idx"])
