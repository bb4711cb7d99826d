"""prox_ffn_noalloc: the decode step with its scratch in a fixed array inside
the library, for callers that cannot allocate device memory while they step
(a serving framework that reserved the device and refuses further
allocations, or a loop where an allocation would synchronise the device).

Collected last on purpose (file name), so that a run stopping at the first
failure has run every other test before this one.  Checks the no-allocation
entry point against prox_ffn on the same layer and input, twice in a row (the
second call finds the first call's scratch contents), within the output bar
the parity tests use; against the oracle's Stage 2 on the GPU's own mask;
that the device memory in use does not change across calls; a layer at the
documented size limit; and that a layer whose scratch would not fit is
rejected before anything is queued."""
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


@pytest.mark.parametrize("d,F,rho,wq", [(1024, 3000, 0.3, 0), (4096, 14336, 0.3, 0),
                                        (1024, 3000, 0.3, 1), (1024, 3000, 0.3, 2)])
def test_no_alloc_matches_prox_ffn_twice(prox, d, F, rho, wq):
    wg, wu, wd = synth.make_weights(d, F, 0.02, 51, device="cuda")
    L = (prox.prox_prepare, prox.prox_prepare_q8, prox.prox_prepare_q4)[wq](wg, wu, wd)
    x = synth.make_x(d, max(1, d // 100), 20.0, 52).cuda()
    y_ref = prox.prox_ffn(L, x, rho).cpu().numpy().astype(np.float64)
    for _ in range(2):
        y = prox.prox_ffn_noalloc(L, x, rho)
        torch.cuda.synchronize()
        assert prox.prox_get_status(L) == 0
        mx, rl = y_errors(y.cpu().numpy(), y_ref)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
        # same mask (deterministic scores), so only the order of the fp32
        # output additions differs
        assert mx <= 1e-5 * max(1.0, float(np.abs(y_ref).max()))
    # a second layer shares the same scratch
    wg2, wu2, wd2 = synth.make_weights(d, F, 0.02, 53, device="cuda")
    L2 = prox.prox_prepare(wg2, wu2, wd2)
    y2_ref = prox.prox_ffn(L2, x, rho).cpu().numpy().astype(np.float64)
    y2 = prox.prox_ffn_noalloc(L2, x, rho)
    torch.cuda.synchronize()
    mx, rl = y_errors(y2.cpu().numpy(), y2_ref)
    assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)


def test_no_alloc_rejects_a_layer_too_large_for_the_scratch(prox):
    d, F = 128, 32768  # proxy partials alone need 4 MiB
    wg, wu, wd = synth.make_weights(d, F, 0.02, 54, device="cuda")
    L = prox.prox_prepare(wg, wu, wd)
    x = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(prox.ProxError) as e:
        prox.prox_ffn_noalloc(L, x, 0.3)
    assert e.value.code == prox.PROX_ERR_UNSUPPORTED_SHAPE


def _oracle_y_on_gpu_mask(prox, L, w_host, x, rho):
    """The oracle's Stage 2 on the channel list the GPU selects for (L, x, rho)
    (the debug entry point: the scores are summed in a fixed order, so every
    entry point selects the same list)."""
    r = prox.prox_ffn_debug(L, x, rho)
    torch.cuda.synchronize()
    idx = r["idx"].cpu().numpy()
    _, y_or = oracle.sparse_ffn(*w_host, host_bits(x.cpu()), idx)
    return y_or


@pytest.mark.parametrize("d,F", [(1024, 3000), (10880, 28544), (8192, 28672)])
def test_no_alloc_matches_the_oracle_and_allocates_nothing(prox, d, F):
    """y against the oracle on the GPU's mask, on a small layer, on one at the
    documented limit (d_ff 28544 at the largest supported d_model, whose
    workspace fills all but ~8 KB of the 4 MiB array, so its last buffers sit
    at the end of the array) and on the Llama-3-70B shape; free device memory
    is the same before and after repeated calls (the first call, which may
    load the library's module and look up the array, comes before the
    measurement)."""
    oracle.build()
    wg, wu, wd = synth.make_weights(d, F, 0.02, 61, device="cuda")
    sizes = prox.prox_query_sizes(d, F)
    assert sizes["workspace"] <= 4 << 20
    L = prox.prox_prepare(wg, wu, wd)
    w_host = tuple(host_bits(t.cpu()) for t in (wg, wu, wd))
    del wg, wu, wd
    x = synth.make_x(d, max(1, d // 100), 20.0, 62).cuda()
    rho = 0.3
    y_or = _oracle_y_on_gpu_mask(prox, L, w_host, x, rho)
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    prox.prox_ffn_noalloc(L, x, rho, y=y)  # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        y.fill_(float("nan"))
        prox.prox_ffn_noalloc(L, x, rho, y=y)
        torch.cuda.synchronize()
        assert prox.prox_get_status(L) == 0
        mx, rl = y_errors(y.cpu().numpy(), y_or)
        assert mx <= ATOL_Y and rl <= RTOL_L2_Y, (mx, rl)
        assert mx <= 1e-3 * max(1.0, float(np.abs(y_or).max()))
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
