"""The C ABI without a GPU: the library builds and loads, exports every
symbol include/prox.h declares, and rejects bad arguments before queueing
any device work (only host-side checks are exercised here)."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "prox.h")


@pytest.fixture(scope="module")
def lib():
    from free_swiglu_ffn_prox_b300 import build, prox

    build.build()
    return prox._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(prox_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "prox_ffn" in names and "prox_prepare" in names and "prox_dense_ffn" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in prox.h but not exported"


def test_only_abi_symbols_are_exported():
    """-fvisibility=hidden: the .so exports the C ABI, not the kernels' C++ names."""
    import subprocess

    from free_swiglu_ffn_prox_b300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.OUT], capture_output=True,
                         text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared_functions()) <= syms
    assert not [s for s in syms if s.startswith("_ZN4prox")]


def test_query_sizes(lib):
    from free_swiglu_ffn_prox_b300 import prox

    s = prox.prox_query_sizes(4096, 14336)
    assert s["proxy_codes"] == 4096 * 14336
    assert s["proxy_scales"] == 32 * 14336 * 4
    assert s["gateup"] == 14336 * 2 * 4096 * 2
    assert s["down_t"] == 14336 * 4096 * 2
    assert s["workspace"] > 0
    s = prox.prox_query_sizes(256, 688)  # ragged d_ff: padded to 704 proxy columns
    assert s["proxy_codes"] == 256 * 704 and s["proxy_scales"] == 2 * 704 * 4
    for d, F in ((100, 64), (0, 64), (256, 0), (16384 + 128, 64), (256, 32769)):
        for q8, q4 in ((False, False), (True, False), (False, True)):
            with pytest.raises(prox.ProxError) as e:
                prox.prox_query_sizes(d, F, q8, q4)
            assert e.value.code == prox.PROX_ERR_UNSUPPORTED_SHAPE


def test_query_sizes_q8(lib):
    """int8 Stage-2 rows: gate|up codes plus 16 bytes of scales per channel,
    W_down^T codes; the proxy and the workspace are those of the bf16 layer."""
    from free_swiglu_ffn_prox_b300 import prox

    for d, F in ((4096, 14336), (256, 688), (8192, 28672)):
        s, s8 = prox.prox_query_sizes(d, F), prox.prox_query_sizes(d, F, q8=True)
        assert s8["gateup"] == F * (2 * d + 16)
        assert s8["down_t"] == F * d
        for n in ("proxy_codes", "proxy_scales", "workspace"):
            assert s8[n] == s[n]


def test_keep_count_agrees_with_oracle(lib):
    from free_swiglu_ffn_prox_b300 import prox

    for n in (1, 7, 256, 688, 4096, 11008, 14336, 28672):
        for f in (1e-7, 0.05, 0.1, 0.3, 0.5, 0.7, 0.999, 1.0):
            assert prox.prox_keep_count(n, f) == oracle.keep_count(n, f)
    assert prox.prox_keep_count(10, 0.0) == 0
    assert prox.prox_keep_count(10, 1.5) == 0
    assert prox.prox_keep_count(10, float("nan")) == 0


def test_status_strings(lib):
    from free_swiglu_ffn_prox_b300 import prox

    for code in range(7):
        assert prox.prox_status_string(code)
    assert prox.prox_status_string(99) == "unknown status"


def test_query_sizes_q4(lib):
    """int4 Stage-2 rows: d / 2 bytes of gate and of up codes plus 16 bytes
    of scales per channel, d / 2 bytes of W_down^T codes; the proxy and the
    workspace are those of the bf16 layer."""
    from free_swiglu_ffn_prox_b300 import prox

    for d, F in ((4096, 14336), (256, 688), (8192, 28672)):
        s, s4 = prox.prox_query_sizes(d, F), prox.prox_query_sizes(d, F, q4=True)
        assert s4["gateup"] == F * (d + 16)
        assert s4["down_t"] == F * d // 2
        for n in ("proxy_codes", "proxy_scales", "workspace"):
            assert s4[n] == s[n]
    with pytest.raises(ValueError):
        prox.prox_query_sizes(256, 688, q8=True, q4=True)


def test_bad_arguments_are_rejected_before_any_device_work(lib):
    vp = ctypes.c_void_p
    h = vp()
    good = [vp(0x10000 + 256 * i) for i in range(8)]  # never dereferenced: checks fail first
    # bad shape
    assert lib.prox_prepare(100, 64, *good, None, ctypes.byref(h)) == 2
    # null pointer
    args = list(good)
    args[2] = None
    assert lib.prox_prepare(256, 64, *args, None, ctypes.byref(h)) == 1
    # misaligned pointer
    args = list(good)
    args[5] = vp(0x10008)
    assert lib.prox_prepare(256, 64, *args, None, ctypes.byref(h)) == 3
    assert lib.prox_prepare(256, 64, *good, None, None) == 1
    # the int8 preparation checks the same way
    assert lib.prox_prepare_q8(100, 64, *good, None, ctypes.byref(h)) == 2
    args = list(good)
    args[6] = None
    assert lib.prox_prepare_q8(256, 64, *args, None, ctypes.byref(h)) == 1
    args = list(good)
    args[6] = vp(0x10004)
    assert lib.prox_prepare_q8(256, 64, *args, None, ctypes.byref(h)) == 3
    assert lib.prox_prepare_q8(256, 64, *good, None, None) == 1
    # and the int4 one
    assert lib.prox_prepare_q4(100, 64, *good, None, ctypes.byref(h)) == 2
    args = list(good)
    args[5] = None
    assert lib.prox_prepare_q4(256, 64, *args, None, ctypes.byref(h)) == 1
    args = list(good)
    args[5] = vp(0x10008)
    assert lib.prox_prepare_q4(256, 64, *args, None, ctypes.byref(h)) == 3
    assert lib.prox_prepare_q4(256, 64, *good, None, None) == 1
    # calls on a null layer
    assert lib.prox_ffn(None, good[0], ctypes.c_float(0.3), good[1], None) == 1
    assert lib.prox_ffn_ex(None, good[0], ctypes.c_float(0.3), ctypes.c_float(0.5), good[1], None) == 1
    assert lib.prox_dense_ffn(None, good[0], good[1], None) == 1
    assert lib.prox_ffn_host(None, good[0], ctypes.c_float(0.3), good[1], None) == 1
    evs = (vp * 5)(*good[:5])
    assert lib.prox_ffn_traced(None, good[0], ctypes.c_float(0.3), ctypes.c_float(0.5), good[1],
                               evs, 5, None) == 1
    assert lib.prox_ffn_blocks(None, good[0], 64, ctypes.c_float(0.3), good[1], None) == 1
    assert lib.prox_ffn_batch(None, good[0], 4, ctypes.c_float(0.3), good[1], None) == 1
    assert lib.prox_ffn_blocks_debug(None, good[0], 64, ctypes.c_float(0.3), good[1], None, None,
                                     None, None) == 1
    assert lib.prox_get_status(None, None) == 1
    assert lib.prox_layer_info(None, None, None) == 1
    assert lib.prox_residual_rmsnorm(256, None, good[1], ctypes.c_float(1e-6), good[2], None) == 1
    assert lib.prox_residual_rmsnorm(256, good[0], good[1], ctypes.c_float(-1.0), good[2], None) == 1
    assert lib.prox_residual_rmsnorm(256, vp(0x10002), good[1], ctypes.c_float(1e-6), good[2], None) == 3
    f = ctypes.c_float
    assert lib.prox_ffn_resnorm(None, good[0], good[1], f(1e-6), good[2], f(0.3), good[3], None) == 1
    lib.prox_destroy(None)  # accepted, no-op


def test_no_alloc_scratch_limit_as_documented(lib):
    """prox_ffn_noalloc's 4 MiB scratch holds the workspace of every d_ff up to
    28544 at any supported d_model (up to 10880); d_ff 28672 up to d_model
    9216, which includes the Llama-3-70B shape; the bounds are exact."""
    from free_swiglu_ffn_prox_b300 import prox

    lim = 4 << 20
    for d in (128, 4096, 8192, 10880):
        assert prox.prox_query_sizes(d, 28544)["workspace"] <= lim
    assert prox.prox_query_sizes(10880, 28608)["workspace"] > lim
    assert prox.prox_query_sizes(9216, 28672)["workspace"] <= lim
    assert prox.prox_query_sizes(9344, 28672)["workspace"] > lim
    with pytest.raises(prox.ProxError):
        prox.prox_query_sizes(11008, 64)  # beyond the supported d_model
    for d, F in ((4096, 11008), (4096, 14336)):
        assert prox.prox_query_sizes(d, F)["workspace"] <= lim
