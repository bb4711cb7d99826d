"""The roofline numerator: bench.py's algorithmic bytes per step must be the
bytes of the library's own layouts that the step reads (sizes from
prox_query_sizes / _q8 / _q4), plus x, y and the lists.  Host only."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def prox():
    from free_swiglu_ffn_prox_b300 import build, prox as p

    build.build()
    return p


@pytest.mark.parametrize("d,F", [(4096, 14336), (4096, 11008), (8192, 28672), (256, 704)])
@pytest.mark.parametrize("rho", [0.5, 0.3, 0.1])
def test_step_bytes_are_the_layout_bytes_the_step_reads(prox, d, F, rho):
    import bench

    kx, k = prox.prox_keep_count(d, 0.5), prox.prox_keep_count(F, rho)
    for wq, fn in ((0, bench.algorithmic_bytes), (1, bench.algorithmic_bytes_q8),
                   (2, bench.algorithmic_bytes_q4)):
        sz = prox.prox_query_sizes(d, F, q8=wq == 1, q4=wq == 2)
        Fp = sz["proxy_codes"] // d            # proxy row length (padded channels)
        assert Fp == F  # these shapes need no padding, so the kept rows are F bytes
        proxy = kx * Fp + sz["proxy_scales"]   # kept proxy rows + every scale
        stage2 = k * (sz["gateup"] // F + sz["down_t"] // F)  # selected rows
        io = 2 * d + 4 * d + 4 * k             # x bf16, y fp32, channel list int32
        assert fn(d, F, k, kx)["step"] == proxy + stage2 + io, (wq, d, F, rho)
        dense = sz["gateup"] + sz["down_t"] + 2 * d + 4 * d
        assert fn(d, F, k, kx)["dense"] == dense, (wq, d, F)


def test_headline_bytes(prox):
    """The 8B layer at keep fraction 0.3: 136,938,292 bytes per step."""
    import bench

    kx, k = prox.prox_keep_count(4096, 0.5), prox.prox_keep_count(14336, 0.3)
    assert (kx, k) == (2048, 4301)
    assert bench.algorithmic_bytes(4096, 14336, k, kx)["step"] == 136_938_292
