"""Batch > 1 decode with per-token masks (prox_ffn_batch), through the C ABI
(marked gpu).  Each token's y must equal the single-token step on that token
(same mask, so only the order of the fp32 output additions differs), and the
oracle's Stage 2 on that token's mask within the parity bar."""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import ATOL_Y, RTOL_L2_Y, host_bits, y_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


@pytest.mark.parametrize("B", [1, 3, 8])
def test_batch_matches_per_token_steps_and_oracle(prox, B):
    d, F, rho = 1024, 3000, 0.3
    wg, wu, wd = synth.make_weights(d, F, 0.02, 91)
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    xs = torch.stack([synth.make_x(d, 10, 20.0, 200 + t) for t in range(B)])
    y = prox.prox_ffn_batch(L, xs.cuda(), rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    for t in range(B):
        r = prox.prox_ffn_debug(L, xs[t].cuda(), rho)
        torch.cuda.synchronize()
        ref = r["y"]
        assert torch.allclose(y[t], ref, rtol=1e-5, atol=1e-6 * float(ref.abs().max()))
        _, y_or = oracle.sparse_ffn(*w, host_bits(xs[t]), r["idx"].cpu().numpy())
        mx, rl = y_errors(y[t].cpu().numpy(), y_or)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (t, mx, rl)


def test_batch_tokens_get_their_own_masks(prox):
    """Two different tokens give two different masks: token 1 of the batch
    equals the single step on token 1, not on token 0."""
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    xs = torch.stack([synth.hidden(shape, seed=s) for s in (1, 2, 3, 4)]).cuda()
    y = prox.prox_ffn_batch(L, xs, 0.3)
    ys = [prox.prox_ffn(L, xs[t], 0.3) for t in range(4)]
    torch.cuda.synchronize()
    assert prox.prox_get_status(L) == 0
    for t in range(4):
        scale = float(ys[t].abs().max())
        assert torch.allclose(y[t], ys[t], rtol=1e-5, atol=1e-6 * scale)
    assert not torch.allclose(ys[0], ys[1], rtol=1e-3, atol=1e-3)


def test_batch_arguments_are_checked(prox):
    d, F = 256, 688
    wg, wu, wd = synth.make_weights(d, F, 0.02, 92, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    x = torch.ones(2, d, dtype=torch.bfloat16, device="cuda")
    lib = prox._load()
    y = torch.empty(2, d, dtype=torch.float32, device="cuda")
    assert lib.prox_ffn_batch(L.handle, prox._ptr(x), 0, 0.3, prox._ptr(y), None) == \
        prox.PROX_ERR_INVALID_ARG
    assert lib.prox_ffn_batch(L.handle, prox._ptr(x), 2, 0.0, prox._ptr(y), None) == \
        prox.PROX_ERR_INVALID_ARG
