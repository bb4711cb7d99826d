"""int8 Stage-2 weights on the GPU vs the oracle, through the C ABI (marked gpu).

prox_prepare_q8 quantizes every Stage-2 row (W_gate[c], W_up[c], W_down[:, c])
symmetrically per row to int8 ("Prox", Abstract: the method composes with
weight quantization).  Bars: codes and scales bit-exact against the oracle's
quantizer; the proxy, and so the channel mask, identical to the bf16 layer's;
y within max-abs 2e-2 and relative-L2 1e-2 (and, for this fp32 path, 1e-3 of
max |y|) of the oracle's int8 Stage 2 evaluated on the GPU's mask, h within
1e-4 relative.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import (ATOL_Y, RTOL_L2_Y, host_bits, tie_band_mask_check, y_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _weights(d, F, seed, sigma=0.02):
    wg, wu, wd = synth.make_weights(d, F, sigma, seed)
    return (wg, wu, wd), (host_bits(wg), host_bits(wu), host_bits(wd))


def _decode_q8(L):
    """(q_gate, s_gate, q_up, s_up, q_down, s_down, tail pad) from the int8 layouts."""
    d, F = L.d_model, L.d_ff
    gu = L.bufs["gateup"].cpu().numpy().reshape(F, 2 * d + 16)
    codes = gu[:, : 2 * d].view(np.int8)
    tail = np.ascontiguousarray(gu[:, 2 * d:]).view(np.float32)  # [F][4]
    qd = L.bufs["down_t"].cpu().numpy().reshape(F, d).view(np.int8)
    return (codes[:, :d], tail[:, 0], codes[:, d:], tail[:, 1], qd, tail[:, 2], tail[:, 3])


def _check_layouts(L, bits):
    q8 = oracle.stage2_q8(*bits)
    qg, sg, qu, su, qd, sd, pad = _decode_q8(L)
    for name, got in (("q_gate", qg), ("q_up", qu), ("q_down", qd)):
        assert np.array_equal(got, q8[name]), name
    for name, got in (("s_gate", sg), ("s_up", su), ("s_down", sd)):
        assert np.array_equal(got.view(np.uint32), q8[name].view(np.uint32)), name
    assert np.all(pad == 0)
    return q8


@pytest.mark.parametrize("d,F", [(256, 688), (128, 64), (384, 1000), (1024, 77), (512, 3000)])
def test_q8_layouts_bit_exact(prox, d, F):
    (wg, wu, wd), bits = _weights(d, F, seed=d + 3 * F)
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    _check_layouts(L8, bits)
    for n in ("proxy_codes", "proxy_scales"):  # the proxy does not change
        assert torch.equal(L8.bufs[n], L.bufs[n]), n


def test_q8_quantizer_edge_rows_on_gpu(prox):
    """All-zero rows (scale 0, codes 0), a row with one nonzero element (its
    code is +-127) and rows whose quotients land on .5 ties."""
    d, F = 256, 64
    (wg, wu, wd), _ = _weights(d, F, seed=5)
    wg[3] = 0.0
    wu[7] = 0.0
    wd[:, 11] = 0.0
    wg[5] = 0.0
    wg[5, 17] = -0.75
    # a row of +-127 and +-0.5 multiples of a power of two: w / s = k + 1/2 exactly
    wu[9] = 0.0
    wu[9, 0] = 127.0 / 64.0
    wu[9, 1:64] = torch.arange(1, 64, dtype=torch.float32).add(0.5).div(64.0).to(torch.bfloat16)
    bits = (host_bits(wg), host_bits(wu), host_bits(wd))
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q8 = _check_layouts(L8, bits)
    assert q8["s_gate"][3] == 0 and not q8["q_gate"][3].any()
    assert q8["s_down"][11] == 0 and not q8["q_down"][11].any()
    assert q8["q_gate"][5, 17] == -127
    assert np.count_nonzero(q8["q_up"][9][1:64] % 2 == 0) == 63  # ties went to even


def _check_q8_step(prox, L8, L, q8, bits, x, rho, kappa=0.5):
    xb = host_bits(x)
    r8 = prox.prox_ffn_debug(L8, x.cuda(), rho, kappa)
    r = prox.prox_ffn_debug(L, x.cuda(), rho, kappa)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L8) == 0 and prox.prox_get_status(L) == 0
    idx = r8["idx"].cpu().numpy()
    # the mask depends on the proxy only: the same as the bf16 layer's, and
    # exact against the oracle outside the tie band
    assert np.array_equal(idx, r["idx"].cpu().numpy())
    kx, k = oracle.keep_count(L.d_model, kappa), oracle.keep_count(L.d_ff, rho)
    kept = oracle.input_topk(xb, kx)
    px = oracle.Proxy(bits[0], bits[1])
    _, _, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    bad, _ = tie_band_mask_check(idx, sc, k)
    assert bad == 0
    h_or, y_or = oracle.sparse_ffn_q8(q8, xb, idx)
    mx, rl = y_errors(r8["y"].cpu().numpy(), y_or)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()), mx
    hh = r8["h"].cpu().numpy().astype(np.float64)
    assert np.allclose(hh, h_or, rtol=1e-4, atol=1e-4 * np.abs(h_or).max())
    # the plain entry point on the int8 layer gives the same y
    y_plain = prox.prox_ffn(L8, x.cuda(), rho) if kappa == 0.5 else None
    if y_plain is not None:
        torch.cuda.synchronize()
        assert torch.allclose(y_plain, r8["y"], rtol=1e-5, atol=1e-6 * float(np.abs(y_or).max()))
    return r8, y_or


@pytest.mark.parametrize("d,F,rho", [(256, 688, 0.5), (128, 64, 0.3), (384, 1000, 0.3),
                                     (1024, 77, 0.5), (512, 3000, 0.05), (2048, 5000, 0.3)])
def test_q8_step_matches_oracle(prox, d, F, rho):
    (wg, wu, wd), bits = _weights(d, F, seed=11 * d + F)
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q8 = oracle.stage2_q8(*bits)
    for s in range(2):
        _check_q8_step(prox, L8, L, q8, bits, synth.make_x(d, max(1, d // 100), 20.0, 50 + s), rho)


def test_q8_keep_fraction_extremes_and_dense(prox):
    d, F = 256, 688
    (wg, wu, wd), bits = _weights(d, F, seed=21)
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q8 = oracle.stage2_q8(*bits)
    x = synth.make_x(d, 4, 20.0, 22)
    r1, _ = _check_q8_step(prox, L8, L, q8, bits, x, 1.0)  # every channel
    _check_q8_step(prox, L8, L, q8, bits, x, 1e-6)         # k = 1
    _check_q8_step(prox, L8, L, q8, bits, x, 0.5, kappa=1e-6)
    y_dense = prox.prox_dense_ffn(L8, x.cuda())
    torch.cuda.synchronize()
    _, y_or = oracle.sparse_ffn_q8(q8, host_bits(x), np.arange(F, dtype=np.int32))
    mx, rl = y_errors(y_dense.cpu().numpy(), y_or)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)
    assert torch.allclose(r1["y"], y_dense, rtol=1e-5, atol=1e-5)


def test_q8_host_buffers(prox):
    d, F = 512, 1500
    (wg, wu, wd), bits = _weights(d, F, seed=31)
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q8 = oracle.stage2_q8(*bits)
    x = synth.make_x(d, 5, 20.0, 32)
    r = prox.prox_ffn_debug(L8, x.cuda(), 0.3)
    y_host = prox.prox_ffn_host(L8, x, 0.3)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L8) == 0
    _, y_or = oracle.sparse_ffn_q8(q8, host_bits(x), r["idx"].cpu().numpy())
    for y in (r["y"], y_host):
        mx, rl = y_errors(y.cpu().numpy(), y_or)
        assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)


def test_q8_full_size_llama3_8b(prox):
    """The Llama-3-8B-shaped layer: layouts bit-exact, and the step at keep
    fraction 0.3 (the measured workload) against the oracle on the GPU's mask."""
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L8 = prox.prox_prepare_q8(wg, wu, wd)
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    bits = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    q8 = _check_layouts(L8, bits)
    x = synth.hidden(shape, seed=1)
    _check_q8_step(prox, L8, L, q8, bits, x, 0.3)


def test_q8_layer_with_block_mask_and_batch(prox):
    """The int8 layer through the block-mask and batch entry points: the
    block mask is the bf16 layer's (it depends on the proxy only), y matches
    the oracle's int8 Stage 2 on it, and a batch equals per-token steps."""
    d, F, bw, rho = 2048, 5000, 8, 0.3
    (wg, wu, wd), bits = _weights(d, F, seed=41)
    L8 = prox.prox_prepare_q8(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q8 = oracle.stage2_q8(*bits)
    x = synth.make_x(d, 20, 20.0, 42)
    r8 = prox.prox_ffn_blocks_debug(L8, x.cuda(), bw, rho)
    r = prox.prox_ffn_blocks_debug(L, x.cuda(), bw, rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L8) == 0 and prox.prox_get_status(L) == 0
    idx = r8["idx"].cpu().numpy()
    assert np.array_equal(idx, r["idx"].cpu().numpy())
    _, y_or = oracle.sparse_ffn_q8(q8, host_bits(x), idx)
    mx, rl = y_errors(r8["y"].cpu().numpy(), y_or)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)
    xs = torch.stack([synth.make_x(d, 20, 20.0, 43 + t) for t in range(3)]).cuda()
    yb = prox.prox_ffn_batch(L8, xs, rho)
    ys = [prox.prox_ffn(L8, xs[t], rho) for t in range(3)]
    torch.cuda.synchronize()
    for t in range(3):
        assert torch.allclose(yb[t], ys[t], rtol=1e-5, atol=1e-6 * float(ys[t].abs().max()))
