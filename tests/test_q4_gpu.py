"""int4 Stage-2 weights on the GPU vs the oracle, through the C ABI (marked gpu).

prox_prepare_q4 quantizes every Stage-2 row (W_gate[c], W_up[c], W_down[:, c])
symmetrically per row to int4 ("Prox", Abstract: the method composes with
weight quantization).  Bars: codes and scales bit-exact against the oracle's
int4 quantizer (unpacked from the nibble layout prox.h states); the proxy,
and so the channel mask, identical to the bf16 layer's; y within max-abs
2e-2 and relative-L2 1e-2 (and, for this fp32 path, 1e-3 of max |y|) of the
oracle's Stage 2 on the int4 codes evaluated on the GPU's mask, h within
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


def _unpack(words):
    """int4 codes from little-endian 32-bit words: element 8 i + 2 m + h of
    a row sits in bits 16 h + 4 m of word i, as n = q + 8."""
    w = np.asarray(words, dtype=np.uint32)
    out = np.empty(w.shape[:-1] + (w.shape[-1] * 8,), dtype=np.int8)
    for m in range(4):
        for h in range(2):
            out[..., 2 * m + h::8] = ((w >> np.uint32(16 * h + 4 * m)) & np.uint32(0xF)).astype(np.int8) - 8
    return out


def _decode_q4(L):
    """(q_gate, s_gate, q_up, s_up, q_down, s_down, tail pad) from the int4 layouts."""
    d, F = L.d_model, L.d_ff
    gu = L.bufs["gateup"].cpu().numpy().reshape(F, d + 16)
    words = np.ascontiguousarray(gu[:, :d]).view(np.uint32)  # [F][d / 4]
    tail = np.ascontiguousarray(gu[:, d:]).view(np.float32)  # [F][4]
    qd = _unpack(L.bufs["down_t"].cpu().numpy().reshape(F, d // 2).view(np.uint32))
    return (_unpack(words[:, : d // 8]), tail[:, 0], _unpack(words[:, d // 8:]), tail[:, 1], qd,
            tail[:, 2], tail[:, 3])


def _check_layouts(L, bits):
    q4 = oracle.stage2_q4(*bits)
    qg, sg, qu, su, qd, sd, pad = _decode_q4(L)
    for name, got in (("q_gate", qg), ("q_up", qu), ("q_down", qd)):
        assert np.array_equal(got, q4[name]), name
    for name, got in (("s_gate", sg), ("s_up", su), ("s_down", sd)):
        assert np.array_equal(got.view(np.uint32), q4[name].view(np.uint32)), name
    assert np.all(pad == 0)
    return q4


def test_unpack_reads_the_stated_nibble_order():
    """The test's own unpacker on a hand-built word: codes -8..7 placed at
    the stated bit positions come back in element order."""
    q = np.array([-8, 7, -1, 0, 3, -3, 5, -6], dtype=np.int64)
    w = 0
    for e in range(8):
        w |= (int(q[e]) + 8) << (16 * (e & 1) + 4 * (e >> 1))
    assert np.array_equal(_unpack(np.array([w], dtype=np.uint32)), q.astype(np.int8))


@pytest.mark.parametrize("d,F", [(256, 688), (128, 64), (384, 1000), (1024, 77), (512, 3000)])
def test_q4_layouts_bit_exact(prox, d, F):
    (wg, wu, wd), bits = _weights(d, F, seed=d + 5 * F)
    L4 = prox.prox_prepare_q4(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    _check_layouts(L4, bits)
    for n in ("proxy_codes", "proxy_scales"):  # the proxy does not change
        assert torch.equal(L4.bufs[n], L.bufs[n]), n


def test_q4_quantizer_edge_rows_on_gpu(prox):
    """All-zero rows (scale 0, codes 0), a row with one nonzero element (its
    code is +-7) and a row whose quotients land on .5 ties."""
    d, F = 256, 64
    (wg, wu, wd), _ = _weights(d, F, seed=7)
    wg[3] = 0.0
    wu[7] = 0.0
    wd[:, 11] = 0.0
    wg[5] = 0.0
    wg[5, 17] = -0.75
    # max 7 / 8 (scale 1 / 8) and quotients k + 1/2 for k = 0..6, both signs
    wu[9] = 0.0
    wu[9, 0] = 7.0 / 8.0
    ties = torch.arange(0, 7, dtype=torch.float32).add(0.5).div(8.0)
    wu[9, 1:8] = ties.to(torch.bfloat16)
    wu[9, 8:15] = (-ties).to(torch.bfloat16)
    bits = (host_bits(wg), host_bits(wu), host_bits(wd))
    L4 = prox.prox_prepare_q4(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q4 = _check_layouts(L4, bits)
    assert q4["s_gate"][3] == 0 and not q4["q_gate"][3].any()
    assert q4["s_down"][11] == 0 and not q4["q_down"][11].any()
    assert q4["q_gate"][5, 17] == -7
    assert np.array_equal(q4["q_up"][9][1:8], [0, 2, 2, 4, 4, 6, 6])    # ties to even
    assert np.array_equal(q4["q_up"][9][8:15], [0, -2, -2, -4, -4, -6, -6])


def _check_q4_step(prox, L4, L, q4, bits, x, rho, kappa=0.5):
    xb = host_bits(x)
    r4 = prox.prox_ffn_debug(L4, x.cuda(), rho, kappa)
    r = prox.prox_ffn_debug(L, x.cuda(), rho, kappa)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L4) == 0 and prox.prox_get_status(L) == 0
    idx = r4["idx"].cpu().numpy()
    assert np.array_equal(idx, r["idx"].cpu().numpy())
    kx, k = oracle.keep_count(L.d_model, kappa), oracle.keep_count(L.d_ff, rho)
    kept = oracle.input_topk(xb, kx)
    px = oracle.Proxy(bits[0], bits[1])
    _, _, sc = oracle.proxy_scores(px.q_gate, px.s_gate, px.q_up, px.s_up, xb, kept)
    bad, _ = tie_band_mask_check(idx, sc, k)
    assert bad == 0
    h_or, y_or = oracle.sparse_ffn_q8(q4, xb, idx)  # the same sums on int4 codes
    mx, rl = y_errors(r4["y"].cpu().numpy(), y_or)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()), mx
    hh = r4["h"].cpu().numpy().astype(np.float64)
    assert np.allclose(hh, h_or, rtol=1e-4, atol=1e-4 * np.abs(h_or).max())
    if kappa == 0.5:
        y_plain = prox.prox_ffn(L4, x.cuda(), rho)
        torch.cuda.synchronize()
        assert torch.allclose(y_plain, r4["y"], rtol=1e-5, atol=1e-6 * float(np.abs(y_or).max()))
    return r4, y_or


@pytest.mark.parametrize("d,F,rho", [(256, 688, 0.5), (128, 64, 0.3), (384, 1000, 0.3),
                                     (1024, 77, 0.5), (512, 3000, 0.05), (2048, 5000, 0.3)])
def test_q4_step_matches_oracle(prox, d, F, rho):
    (wg, wu, wd), bits = _weights(d, F, seed=13 * d + F)
    L4 = prox.prox_prepare_q4(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q4 = oracle.stage2_q4(*bits)
    for s in range(2):
        _check_q4_step(prox, L4, L, q4, bits, synth.make_x(d, max(1, d // 100), 20.0, 60 + s), rho)


def test_q4_keep_fraction_extremes_and_dense(prox):
    d, F = 256, 688
    (wg, wu, wd), bits = _weights(d, F, seed=23)
    L4 = prox.prox_prepare_q4(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q4 = oracle.stage2_q4(*bits)
    x = synth.make_x(d, 4, 20.0, 24)
    r1, _ = _check_q4_step(prox, L4, L, q4, bits, x, 1.0)  # every channel
    _check_q4_step(prox, L4, L, q4, bits, x, 1e-6)         # k = 1
    _check_q4_step(prox, L4, L, q4, bits, x, 0.5, kappa=1e-6)
    y_dense = prox.prox_dense_ffn(L4, x.cuda())
    torch.cuda.synchronize()
    _, y_or = oracle.sparse_ffn_q8(q4, host_bits(x), np.arange(F, dtype=np.int32))
    mx, rl = y_errors(y_dense.cpu().numpy(), y_or)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)
    assert torch.allclose(r1["y"], y_dense, rtol=1e-5, atol=1e-5)


def test_q4_full_size_llama3_8b(prox):
    """The Llama-3-8B-shaped layer: layouts bit-exact, and the step at keep
    fraction 0.3 (the measured workload) against the oracle on the GPU's
    mask, through device and host buffers."""
    shape = synth.LLAMA3_8B
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L4 = prox.prox_prepare_q4(wg, wu, wd)
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    bits = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    q4 = _check_layouts(L4, bits)
    x = synth.hidden(shape, seed=1)
    r4, y_or = _check_q4_step(prox, L4, L, q4, bits, x, 0.3)
    y_host = prox.prox_ffn_host(L4, x, 0.3)
    mx, rl = y_errors(y_host.numpy(), y_or)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)


def test_q4_layer_with_block_mask_stack_and_batch(prox):
    """The int4 layer through the block-mask, stack and batch entry points:
    the block mask is the bf16 layer's, y matches the oracle's Stage 2 on
    the int4 codes, a two-layer stack equals its per-layer steps, and a
    batch equals per-token steps."""
    d, F, bw, rho = 2048, 5000, 8, 0.3
    (wg, wu, wd), bits = _weights(d, F, seed=45)
    L4 = prox.prox_prepare_q4(wg.cuda(), wu.cuda(), wd.cuda())
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    q4 = oracle.stage2_q4(*bits)
    x = synth.make_x(d, 20, 20.0, 46)
    r4 = prox.prox_ffn_blocks_debug(L4, x.cuda(), bw, rho)
    r = prox.prox_ffn_blocks_debug(L, x.cuda(), bw, rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L4) == 0 and prox.prox_get_status(L) == 0
    idx = r4["idx"].cpu().numpy()
    assert np.array_equal(idx, r["idx"].cpu().numpy())
    _, y_or = oracle.sparse_ffn_q8(q4, host_bits(x), idx)
    mx, rl = y_errors(r4["y"].cpu().numpy(), y_or)
    assert mx <= 1e-3 * max(1.0, np.abs(y_or).max()) and rl <= RTOL_L2_Y, (mx, rl)
    xs_st, ys_st = prox.prox_stack_ffn([L4, L4], x.cuda(), rho)
    y0 = prox.prox_ffn(L4, x.cuda(), rho)
    y1 = prox.prox_ffn(L4, xs_st[1], rho)
    torch.cuda.synchronize()
    assert prox.prox_get_status(L4) == 0
    for got, want in ((ys_st[0], y0), (ys_st[1], y1)):
        assert torch.allclose(got, want, rtol=1e-5, atol=1e-6 * float(want.abs().max()))
    xs = torch.stack([synth.make_x(d, 20, 20.0, 47 + t) for t in range(3)]).cuda()
    yb = prox.prox_ffn_batch(L4, xs, rho)
    ys = [prox.prox_ffn(L4, xs[t], rho) for t in range(3)]
    torch.cuda.synchronize()
    for t in range(3):
        assert torch.allclose(yb[t], ys[t], rtol=1e-5, atol=1e-6 * float(ys[t].abs().max()))
    with pytest.raises(prox.ProxError):  # union batches take bf16 rows only
        prox.prox_ffn_batch_union(L4, xs, rho)
