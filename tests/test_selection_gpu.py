"""The exact channel top-k under heavy ties and crowded score bins, at the
Llama-3-8B layer size, through the C ABI (marked gpu).

The selection ranks channels by the bit pattern of their fp32 score (the
"magnitude ranking" of the intermediate state, Prox abstract), ties to the
lower channel.  It resolves the k-th key digit by digit; the first digit is
the top 11 bits of the key.  Two inputs stress the paths a random layer
never takes:
  * x = 0: every score is 0, all F keys tie, so the k selected channels are
    the first k and y = 0;
  * a crowded layer: every channel's gate and up rows are one shared row plus
    5% independent noise, so the proxy scores crowd together and more than
    2048 distinct keys share the k-th key's first digit.
Bars as in the other parity tests (the kept inputs exact, the mask exact
outside the tie band, y within max-abs 2e-2 and relative-L2 1e-2 on the
GPU's mask), for the channel mask and for block-granular masks.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import TIE_BAND, check_step, host_bits

pytestmark = pytest.mark.gpu

D, F = 4096, 14336


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _crowded_weights(noise=0.05, seed=7):
    g = torch.Generator().manual_seed(seed)
    base_g = torch.randn(D, generator=g) * 0.02
    base_u = torch.randn(D, generator=g) * 0.02
    wg = (base_g + noise * 0.02 * torch.randn(F, D, generator=g)).to(torch.bfloat16)
    wu = (base_u + noise * 0.02 * torch.randn(F, D, generator=g)).to(torch.bfloat16)
    wd = (torch.randn(D, F, generator=g) * 0.02).to(torch.bfloat16)
    return wg, wu, wd


def _first_digit_crowd(scores, k):
    """(keys sharing the k-th key's first 11-bit digit, distinct keys among them)."""
    key = np.ascontiguousarray(scores, dtype=np.float32).view(np.uint32)
    kth = np.sort(key)[::-1][k - 1]
    same = key[(key >> 20) == (kth >> 20)]
    return int(same.size), int(np.unique(same).size)


@pytest.fixture(scope="module")
def crowded(prox):
    wg, wu, wd = _crowded_weights()
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    return L, w, oracle.Proxy(w[0], w[1])


def test_all_scores_tied_at_full_size(prox):
    wg, wu, wd = synth.make_weights(D, F, 0.02, 81, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    x = torch.zeros(D, dtype=torch.bfloat16, device="cuda")
    for rho in (0.5, 0.3, 0.1):
        r = prox.prox_ffn_debug(L, x, rho)
        torch.cuda.synchronize()
        assert prox.prox_get_status(L) == 0
        k = oracle.keep_count(F, rho)
        sc = r["scores"].cpu().numpy()
        assert np.all(sc == 0.0)
        assert _first_digit_crowd(sc, k)[0] == F  # every key in one bin
        assert np.array_equal(r["idx"].cpu().numpy(), np.arange(k))
        assert np.array_equal(r["kept"].cpu().numpy(), np.arange(D // 2))
        assert torch.count_nonzero(r["y"]) == 0
        y = prox.prox_ffn(L, x, rho)
        torch.cuda.synchronize()
        assert torch.count_nonzero(y) == 0
    for bw in (16, 64):
        r = prox.prox_ffn_blocks_debug(L, x, bw, 0.3)
        torch.cuda.synchronize()
        K = oracle.keep_count(F // bw, 0.3)
        assert np.array_equal(r["idx"].cpu().numpy(), np.arange(K * bw))
        assert torch.count_nonzero(r["y"]) == 0
    assert prox.prox_get_status(L) == 0


@pytest.mark.parametrize("rho", [0.5, 0.3, 0.1])
def test_crowded_first_digit_at_full_size(prox, crowded, rho):
    L, w, px = crowded
    x = synth.make_x(D, 41, 20.0, 3)
    r = check_step(prox, L, w, x, rho, px=px)
    n_same, n_distinct = _first_digit_crowd(r["scores"].cpu().numpy(), r["k"])
    if rho == 0.3:
        # the case this layer is built for: the k-th key's first digit is shared
        # by more than 2048 keys, nearly all distinct
        assert n_same > 2048 and n_distinct > 2048, (n_same, n_distinct)


@pytest.mark.parametrize("bw", [16, 64])
def test_crowded_block_mask_at_full_size(prox, crowded, bw):
    """Block sums of crowded channel scores crowd as well; the block mask
    stays exact outside the tie band of the K-th block sum."""
    L, w, px = crowded
    x = synth.make_x(D, 41, 20.0, 3)
    xb = host_bits(x)
    r = prox.prox_ffn_blocks_debug(L, x.cuda(), bw, 0.3)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    E = F // bw
    K = oracle.keep_count(E, 0.3)
    kept = oracle.input_topk(xb, oracle.keep_count(D, 0.5))
    _, _, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    idx = r["idx"].cpu().numpy()
    assert idx.size == K * bw and np.all(np.diff(idx) > 0)
    blk = idx.reshape(K, bw)
    assert np.all(blk[:, 0] % bw == 0) and np.all(blk == blk[:, :1] + np.arange(bw))
    got = set((blk[:, 0] // bw).tolist())
    idx_or, S = oracle.block_topk(sc, bw, K)
    want = set((idx_or.reshape(K, bw)[:, 0] // bw).tolist())
    SK = np.sort(S)[::-1][K - 1]
    band = np.abs(S - SK) <= TIE_BAND * abs(SK)
    assert all((e in got) == (e in want) for e in range(E) if not band[e])
    _, y_or = oracle.sparse_ffn(*w, xb, idx)
    y = r["y"].cpu().numpy().astype(np.float64)
    assert np.abs(y - y_or).max() <= 1e-3 * max(1.0, np.abs(y_or).max())
