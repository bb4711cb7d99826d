"""GPU vs oracle parity through the C ABI (marked gpu).

Bars: proxy codes/scales and the kept-input set bit-exact; the channel mask
exact outside the tie band (channels whose oracle score lies within 1e-4
relative of the oracle's k-th score may differ); y within max-abs 2e-2 and
relative-L2 1e-2 of the oracle's sparse FFN evaluated on the GPU's mask.
"""
import numpy as np
import pytest
import torch

import oracle
from free_swiglu_ffn_prox_b300 import synth
from parity_util import (ATOL_Y, RTOL_L2_Y, TIE_BAND, check_step, decode_proxy, host_bits,
                         tie_band_mask_check, y_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prox():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


def _layer(prox, d, F, sigma=0.02, seed=0, device="cpu"):
    wg, wu, wd = synth.make_weights(d, F, sigma, seed, device=device)
    L = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    torch.cuda.synchronize()
    return L, (host_bits(wg), host_bits(wu), host_bits(wd))


def _x(d, n_out, seed):
    return synth.make_x(d, n_out, 20.0, seed)


def _check_step(prox, L, w, x, rho, kappa=0.5, px=None):
    return check_step(prox, L, w, x, rho, kappa, px)


@pytest.mark.parametrize("d,F", [(256, 688), (128, 64), (384, 1000), (1024, 77), (512, 3000)])
def test_prepare_layouts_bit_exact(prox, d, F):
    L, (wg, wu, wd) = _layer(prox, d, F, seed=d + F)
    qg, qu, sg, su, pad_codes, pad_scales = decode_proxy(L)
    og, osg = oracle.quantize(wg)
    ou, osu = oracle.quantize(wu)
    assert np.array_equal(qg, og) and np.array_equal(qu, ou)
    assert np.array_equal(sg, osg) and np.array_equal(su, osu)
    assert np.all(pad_codes == 0x88) and np.all(pad_scales == 0)
    gu = L.bufs["gateup"].cpu().view(torch.int16).numpy().view(np.uint16).reshape(F, 2, d)
    assert np.array_equal(gu[:, 0, :], wg) and np.array_equal(gu[:, 1, :], wu)
    dt = L.bufs["down_t"].cpu().view(torch.int16).numpy().view(np.uint16).reshape(F, d)
    assert np.array_equal(dt, wd.T)


@pytest.mark.parametrize("d,F,rho", [(256, 688, 0.5), (256, 688, 0.1), (128, 64, 0.3),
                                     (384, 1000, 0.3), (1024, 77, 0.5), (512, 3000, 0.05),
                                     (2048, 5000, 0.3)])
def test_prox_ffn_matches_oracle(prox, d, F, rho):
    L, w = _layer(prox, d, F, seed=7 * d + F)
    for s in range(3):
        _check_step(prox, L, w, _x(d, max(1, d // 100), seed=100 + s), rho)


def test_keep_fraction_extremes(prox):
    d, F = 256, 688
    L, w = _layer(prox, d, F, seed=3)
    x = _x(d, 4, seed=9)
    r1 = _check_step(prox, L, w, x, 1.0)
    assert r1["k"] == F
    y_dense = prox.prox_dense_ffn(L, x.cuda())
    torch.cuda.synchronize()
    assert torch.allclose(r1["y"], y_dense, rtol=1e-5, atol=1e-5)
    _check_step(prox, L, w, x, 1e-6)  # k = 1
    _check_step(prox, L, w, x, 0.5, kappa=1.0)   # every input kept
    _check_step(prox, L, w, x, 0.5, kappa=1e-6)  # a single input kept


def test_dense_matches_oracle(prox):
    for d, F in ((256, 688), (1024, 2000)):
        L, (wg, wu, wd) = _layer(prox, d, F, seed=11)
        x = _x(d, 4, seed=12)
        y = prox.prox_dense_ffn(L, x.cuda())
        torch.cuda.synchronize()
        _, y_or = oracle.dense_ffn(wg, wu, wd, host_bits(x))
        mx, rl = y_errors(y.cpu().numpy(), y_or)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y


def test_degenerate_inputs(prox):
    d, F = 256, 300
    L, w = _layer(prox, d, F, seed=5)
    # x = 0: every score is 0, ties -> the first k channels, y = 0
    x0 = torch.zeros(d, dtype=torch.bfloat16)
    r = prox.prox_ffn_debug(L, x0.cuda(), 0.3)
    torch.cuda.synchronize()
    k = oracle.keep_count(F, 0.3)
    assert np.array_equal(r["idx"].cpu().numpy(), np.arange(k))
    assert np.array_equal(r["kept"].cpu().numpy(), np.arange(d // 2))
    assert torch.count_nonzero(r["y"]) == 0
    # one-hot and heavily tied inputs
    xo = torch.zeros(d, dtype=torch.bfloat16)
    xo[77] = -3.5
    _check_step(prox, L, w, xo, 0.3)
    xt = torch.tensor(np.random.default_rng(1).choice([0.0, -1.0, 1.0, 2.0], size=d),
                      dtype=torch.float32).to(torch.bfloat16)
    _check_step(prox, L, w, xt, 0.3)


def test_channel_permutation_identity_on_gpu(prox):
    """Eq. (2) of the PrunePath page: permuting channels of all three weights
    permutes the mask and leaves y unchanged (up to fp32 rounding)."""
    d, F = 512, 1024
    wg, wu, wd = synth.make_weights(d, F, 0.02, 21)
    perm = torch.randperm(F, generator=torch.Generator().manual_seed(2))
    L1 = prox.prox_prepare(wg.cuda(), wu.cuda(), wd.cuda())
    L2 = prox.prox_prepare(wg[perm].contiguous().cuda(), wu[perm].contiguous().cuda(),
                           wd[:, perm].contiguous().cuda())
    x = _x(d, 5, 22).cuda()
    r1 = prox.prox_ffn_debug(L1, x, 0.3)
    r2 = prox.prox_ffn_debug(L2, x, 0.3)
    torch.cuda.synchronize()
    s1 = r1["scores"].cpu()
    s2 = r2["scores"].cpu()
    assert torch.allclose(s1[perm], s2, rtol=1e-5, atol=1e-6)
    assert torch.allclose(r1["y"], r2["y"], rtol=1e-4, atol=1e-4)


def test_errors_are_reported_not_raised_on_device(prox):
    L, _ = _layer(prox, 256, 688, seed=1)
    x = torch.zeros(256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn(L, x, 0.0)
    assert e.value.code == prox.PROX_ERR_INVALID_ARG
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn(L, x, 1.5)
    assert e.value.code == prox.PROX_ERR_INVALID_ARG
    buf = torch.zeros(300, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn(L, buf[1:257], 0.3)
    assert e.value.code == prox.PROX_ERR_MISALIGNED
    assert prox.prox_get_status(L) == 0


def test_host_buffer_and_traced_entry_points(prox):
    """prox_ffn_host (host x/y, copies queued by the library) and
    prox_ffn_traced (events between the kernels) compute what prox_ffn does."""
    d, F = 1024, 3000
    L, (wg, wu, wd) = _layer(prox, d, F, seed=31)
    x = _x(d, 10, 32)
    y_dev = prox.prox_ffn(L, x.cuda(), 0.3)
    xh = x.clone().pin_memory()
    yh = torch.full((d,), float("nan")).pin_memory()
    prox.prox_ffn_host(L, xh, 0.3, y_host=yh)
    torch.cuda.synchronize()
    assert torch.allclose(yh, y_dev.cpu(), rtol=1e-5, atol=1e-5)
    y_pageable = prox.prox_ffn_host(L, x.clone(), 0.3)  # pageable memory works too
    torch.cuda.synchronize()
    assert torch.allclose(y_pageable, y_dev.cpu(), rtol=1e-5, atol=1e-5)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(prox.PROX_TRACE_EVENTS)]
    for e in evs:
        e.record()
    y_tr = prox.prox_ffn_traced(L, x.cuda(), 0.3, evs)
    torch.cuda.synchronize()
    assert torch.allclose(y_tr, y_dev, rtol=1e-5, atol=1e-5)
    dt = [evs[i].elapsed_time(evs[i + 1]) for i in range(prox.PROX_TRACE_EVENTS - 1)]
    assert all(t >= 0.0 for t in dt) and sum(dt) > 0.0
    with pytest.raises(prox.ProxError):
        prox.prox_ffn_host(L, xh, 1.5, y_host=yh)
    # the same traced step captured in a CUDA graph (event nodes)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    y_g = torch.empty(d, device="cuda")
    xg = x.cuda()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            prox.prox_ffn_traced(L, xg, 0.3, evs, y=y_g)
    g.replay()
    torch.cuda.synchronize()
    assert torch.allclose(y_g, y_dev, rtol=1e-5, atol=1e-5)
    dt = [evs[i].elapsed_time(evs[i + 1]) for i in range(prox.PROX_TRACE_EVENTS - 1)]
    assert all(t >= 0.0 for t in dt)
    assert prox.prox_get_status(L) == 0


def test_bounded_barrier_wait_reports_timeout_and_recovers(prox):
    """Failure detection without a GPU fault: one CTA withholds its arrival
    at a grid barrier, the others give up after 20 ms and record
    PROX_ERR_TIMEOUT; the status read resets the barrier and the next step on
    the same layer is correct again."""
    d, F = 512, 1500
    L, w = _layer(prox, d, F, seed=41)
    x = _x(d, 5, 42)
    _check_step(prox, L, w, x, 0.3)
    assert prox.prox_test_barrier_timeout(L, x.cuda()) == prox.PROX_ERR_TIMEOUT
    assert prox.prox_get_status(L) == 0
    _check_step(prox, L, w, x, 0.3)
    _check_step(prox, L, w, _x(d, 5, 43), 0.1)


def test_masks_are_deterministic(prox):
    """The proxy partials are summed in a fixed order, so repeated steps give
    the same scores and the same channel list bit for bit."""
    d, F = 4096, 14336
    wg, wu, wd = synth.make_weights(d, F, 0.02, 5, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    x = _x(d, 41, 6).cuda()
    r1 = prox.prox_ffn_debug(L, x, 0.3)
    r2 = prox.prox_ffn_debug(L, x, 0.3)
    torch.cuda.synchronize()
    assert torch.equal(r1["scores"], r2["scores"])
    assert torch.equal(r1["idx"], r2["idx"])
    assert torch.equal(r1["kept"], r2["kept"])
    assert torch.allclose(r1["y"], r2["y"], rtol=0, atol=1e-5 * float(r1["y"].abs().max()))


# ------------------------------------------------------------- full-size layers
FULL = [synth.LLAMA2_7B, synth.LLAMA3_8B, synth.LLAMA3_70B]


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_layers(prox, shape):
    """The Llama-shaped layers at every keep fraction: kept inputs exact,
    mask exact outside the tie band against the oracle's full proxy, y within
    the bar against the oracle's Stage 2 on the GPU's mask."""
    wg, wu, wd = synth.layer(shape, seed=0, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    torch.cuda.synchronize()
    w = (host_bits(wg), host_bits(wu), host_bits(wd))
    del wg, wu, wd
    qg, qu, sg, su, _, _ = decode_proxy(L)
    px = oracle.Proxy.__new__(oracle.Proxy)
    px.q_gate, px.s_gate = oracle.quantize(w[0])
    px.q_up, px.s_up = oracle.quantize(w[1])
    assert np.array_equal(qg, px.q_gate) and np.array_equal(qu, px.q_up)
    assert np.array_equal(sg, px.s_gate) and np.array_equal(su, px.s_up)
    x = synth.hidden(shape, seed=1)
    for rho in shape.keep_fractions:
        _check_step(prox, L, w, x, rho, px=px)


# ------------------------------------------------------------- stack glue
def _bf16_ulp_diff(a_bits, b_bits):
    """|a - b| in units of the larger bf16 ulp of the pair (both finite)."""
    a = oracle.bf16_bits_to_f64(a_bits)
    b = oracle.bf16_bits_to_f64(b_bits)
    m = np.maximum(np.abs(a), np.abs(b))
    ulp = np.where(m > 0, 2.0 ** (np.floor(np.log2(np.maximum(m, 1e-300))) - 7), 1.0)
    return np.abs(a - b) / ulp


@pytest.mark.parametrize("d", [128, 1000, 4096, 8192, 16384])
def test_residual_rmsnorm_matches_oracle(prox, d):
    """x_next = bf16(RMSNorm(x + y)): the fp32 kernel and the fp64 oracle
    round to the same bf16 except where the exact value sits next to a
    rounding midpoint, where they may differ by one ulp."""
    x = _x(d, max(1, d // 100), seed=d)
    y = torch.randn(d, generator=torch.Generator().manual_seed(d + 1)) * 9.0
    out = prox.prox_residual_rmsnorm(x.cuda(), y.cuda())
    torch.cuda.synchronize()
    got = host_bits(out)
    ref = oracle.residual_rmsnorm(host_bits(x), y.double().numpy())
    ulps = _bf16_ulp_diff(got, ref)
    assert ulps.max() <= 1.0
    assert np.count_nonzero(got != ref) <= max(2, d // 500)
    # eps dominates an all-zero residual: the output is exactly zero
    z = prox.prox_residual_rmsnorm(torch.zeros(d, dtype=torch.bfloat16, device="cuda"),
                                   torch.zeros(d, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(z) == 0


def test_short_stack_matches_oracle_layer_by_layer(prox):
    """Four stacked layers, x_{l+1} = RMSNorm(x_l + y_l) on the GPU: every
    layer's step is checked against the oracle on the GPU's own x_l (so a
    tie-band mask difference in one layer does not propagate into the next
    comparison), and each glue step against the oracle's glue."""
    d, F = 1024, 2816
    x = _x(d, 10, seed=70).cuda()
    for l in range(4):
        L, w = _layer(prox, d, F, seed=1000 + l)
        r = _check_step(prox, L, w, x.cpu(), 0.3)
        y = prox.prox_ffn(L, x, 0.3)
        torch.cuda.synchronize()
        x_next = prox.prox_residual_rmsnorm(x, y)
        torch.cuda.synchronize()
        ref = oracle.residual_rmsnorm(host_bits(x), y.cpu().double().numpy())
        assert _bf16_ulp_diff(host_bits(x_next), ref).max() <= 1.0
        assert torch.allclose(y, r["y"], rtol=0, atol=1e-5 * float(y.abs().max()))
        x = x_next


def test_fused_stack_glue_matches_the_separate_glue_and_the_oracle(prox):
    """prox_ffn_resnorm computes x = bf16(RMSNorm(x_prev + y_prev)) inside the
    step: x_out is the oracle's glue to within one bf16 ulp (in every CTA the
    same value: the mask and y then match the oracle as for prox_ffn), and the
    step on it matches the oracle layer by layer."""
    d, F = 1024, 2816
    L0, _ = _layer(prox, d, F, seed=1200)
    x = _x(d, 10, seed=72).cuda()
    y = prox.prox_ffn(L0, x, 0.3)
    torch.cuda.synchronize()
    for l in range(1, 4):
        L, w = _layer(prox, d, F, seed=1200 + l)
        x_out, y_next = prox.prox_ffn_resnorm(L, x, y, 0.3)
        torch.cuda.synchronize()
        assert prox.prox_get_status(L) == 0
        ref = oracle.residual_rmsnorm(host_bits(x), y.cpu().double().numpy())
        assert _bf16_ulp_diff(host_bits(x_out), ref).max() <= 1.0
        sep = prox.prox_residual_rmsnorm(x, y)
        torch.cuda.synchronize()
        assert _bf16_ulp_diff(host_bits(x_out), host_bits(sep)).max() <= 1.0
        r = _check_step(prox, L, w, x_out.cpu(), 0.3)
        assert torch.allclose(y_next, r["y"], rtol=0, atol=1e-5 * float(y_next.abs().max()))
        x, y = x_out, y_next
    # outputs may not overlap the inputs (CTA 0 writes them while all CTAs read)
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn_resnorm(L, x, y, 0.3, x_out=x)
    assert e.value.code == prox.PROX_ERR_INVALID_ARG
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn_resnorm(L, x, y, 0.3, y=y)
    assert e.value.code == prox.PROX_ERR_INVALID_ARG
