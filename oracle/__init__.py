"""CPU oracle for the Prox sparse SwiGLU FFN decode step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``prox_oracle.c`` (plain C, fp64); this module builds
it with gcc and marshals numpy arrays through ctypes.  Inputs are raw bf16 bit
patterns (``numpy.uint16``) in nn.Linear layouts: ``W_gate``/``W_up`` are
``[F][d]`` and ``W_down`` is ``[d][F]``.

Page citations (by title and section):
  * Prox: Training-Free FFN Activation Sparsity via Approximate
    Intermediate-Channel Salience in LLMs -- Abstract (two-stage method).
  * PrunePath: Towards Highly Structured Sparse Language Models --
    Sec. 2.1 Eq. (1) (SwiGLU FFN), Sec. 2.2 Eq. (2) (channel permutation
    identity, used by the tests as an invariant).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "prox_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32 = ctypes.c_int
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile prox_oracle.c into liboracle.so next to it (gcc, no fast-math,
    no FMA contraction so the binary32 quantizer steps round as written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_fp16_to_double.restype = ctypes.c_double
            lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_round_to_fp16.restype = ctypes.c_double
            lib.oracle_round_to_fp16.argtypes = [ctypes.c_float]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_keep_count.restype = _i32
            lib.oracle_keep_count.argtypes = [_i32, ctypes.c_float]
            lib.oracle_quantize.argtypes = [_i32, _i32, _ptr, _ptr, _ptr]
            lib.oracle_input_topk.argtypes = [_i32, _ptr, _i32, _ptr]
            lib.oracle_proxy_scores.argtypes = [_i32, _i32] + [_ptr] * 5 + [_i32] + [_ptr] * 4
            lib.oracle_channel_topk.argtypes = [_i32, _ptr, _i32, _ptr]
            lib.oracle_sparse_ffn.argtypes = [_i32, _i32] + [_ptr] * 4 + [_i32] + [_ptr] * 3
            lib.oracle_dense_ffn.argtypes = [_i32, _i32] + [_ptr] * 6
            lib.oracle_prox_ffn.argtypes = [_i32, _i32] + [_ptr] * 8 + [_i32, _i32] + [_ptr] * 5
            lib.oracle_residual_rmsnorm.argtypes = [_i32, _ptr, _ptr, ctypes.c_double, _ptr]
            lib.oracle_quantize_rows_q8.argtypes = [_i32, _i32, _ptr, _ptr, _ptr]
            lib.oracle_sparse_ffn_q8.argtypes = [_i32, _i32] + [_ptr] * 7 + [_i32, _ptr, _ptr, _ptr]
            lib.oracle_quantize_rows_q4.argtypes = [_i32, _i32, _ptr, _ptr, _ptr]
            lib.oracle_block_topk.argtypes = [_i32, _ptr, _i32, _i32, _ptr, _ptr]
            lib.oracle_contrib_scores.argtypes = [_i32, _i32, _ptr, _ptr, _ptr]
            for name in ("oracle_quantize", "oracle_input_topk", "oracle_proxy_scores",
                         "oracle_channel_topk", "oracle_sparse_ffn", "oracle_dense_ffn",
                         "oracle_prox_ffn", "oracle_residual_rmsnorm", "oracle_quantize_rows_q8",
                         "oracle_sparse_ffn_q8", "oracle_block_topk", "oracle_contrib_scores",
                         "oracle_quantize_rows_q4"):
                getattr(lib, name).restype = _i32
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: bad arguments (rc={rc})")


# ---------------------------------------------------------------- formats
def bf16_to_double(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(v)) for v in b]).reshape(np.shape(bits))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Vectorised bf16 decode (the pattern is the top half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp16_to_double(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_fp16_to_double(int(v)) for v in b]).reshape(np.shape(bits))


def round_to_fp16(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_round_to_fp16(float(t)) for t in v]).reshape(np.shape(values))


def double_to_bf16(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib.oracle_double_to_bf16(float(t)) for t in v],
                    dtype=np.uint16).reshape(np.shape(values))


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


def keep_count(n: int, frac: float) -> int:
    return int(_load().oracle_keep_count(int(n), float(np.float32(frac))))


# ---------------------------------------------------------------- the method
def quantize(w_bits: np.ndarray):
    """a0: int4 group-128 symmetric proxy codes q[F][d] and fp16 scales s[F][G]."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    F, d = w.shape
    q = np.empty((F, d), dtype=np.int8)
    s = np.empty((F, d // 128), dtype=np.float64)
    _check(lib.oracle_quantize(F, d, _p(w), _p(q), _p(s)), "quantize")
    return q, s


def input_topk(x_bits: np.ndarray, kx: int) -> np.ndarray:
    """a1: ascending indices of the kx largest |x_j| (ties -> lower j)."""
    lib = _load()
    x = _c(x_bits, np.uint16).ravel()
    kept = np.empty(kx, dtype=np.int32)
    _check(lib.oracle_input_topk(x.size, _p(x), int(kx), _p(kept)), "input_topk")
    return kept


def proxy_scores(q_gate, s_gate, q_up, s_up, x_bits, kept):
    """a2: (g~, u~, score) in fp64 over the kept inputs."""
    lib = _load()
    qg, qu = _c(q_gate, np.int8), _c(q_up, np.int8)
    sg, su = _c(s_gate, np.float64), _c(s_up, np.float64)
    x = _c(x_bits, np.uint16).ravel()
    kept = _c(kept, np.int32)
    F, d = qg.shape
    g = np.empty(F)
    u = np.empty(F)
    sc = np.empty(F)
    _check(lib.oracle_proxy_scores(F, d, _p(qg), _p(sg), _p(qu), _p(su), _p(x), kept.size,
                                   _p(kept), _p(g), _p(u), _p(sc)), "proxy_scores")
    return g, u, sc


def contrib_scores(state_score, w_down_bits) -> np.ndarray:
    """Second selection signal (COUNTDOWN reading): |h~_c| * ||W_down[:, c]||_2,
    the magnitude of channel c's term of the down projection's linear
    combination, from the proxy state score |h~_c| (fp64)."""
    lib = _load()
    sc = _c(state_score, np.float64).ravel()
    wd = _c(w_down_bits, np.uint16)
    d, F = wd.shape
    if sc.size != F:
        raise ValueError("state_score must have d_ff entries")
    out = np.empty(F)
    _check(lib.oracle_contrib_scores(F, d, _p(wd), _p(sc), _p(out)), "contrib_scores")
    return out


def channel_topk(score: np.ndarray, k: int) -> np.ndarray:
    """a3: ascending indices of the k largest scores (ties -> lower channel)."""
    lib = _load()
    sc = _c(score, np.float64)
    idx = np.empty(k, dtype=np.int32)
    _check(lib.oracle_channel_topk(sc.size, _p(sc), int(k), _p(idx)), "channel_topk")
    return idx


def block_topk(score: np.ndarray, bw: int, K: int):
    """f3: channels of the K blocks of bw contiguous channels whose summed
    score is largest (ties -> lower block), ascending; returns (idx, S[E])."""
    lib = _load()
    sc = _c(score, np.float64).ravel()
    E = sc.size // int(bw) if bw > 0 else 0
    idx = np.empty(max(int(K), 0) * max(int(bw), 0), dtype=np.int32)
    S = np.empty(max(E, 1))
    _check(lib.oracle_block_topk(sc.size, _p(sc), int(bw), int(K), _p(S), _p(idx)),
           "block_topk")
    return idx, S[:E]


def sparse_ffn(w_gate, w_up, w_down, x_bits, idx):
    """a4-a5: Stage 2 on the channel list idx -> (h[len(idx)], y[d]) in fp64."""
    lib = _load()
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    x = _c(x_bits, np.uint16).ravel()
    idx = _c(idx, np.int32).ravel()
    F, d = wg.shape
    h = np.empty(idx.size)
    y = np.empty(d)
    _check(lib.oracle_sparse_ffn(F, d, _p(wg), _p(wu), _p(wd), _p(x), idx.size,
                                 _p(idx) if idx.size else None, _p(h), _p(y)), "sparse_ffn")
    return h, y


def dense_ffn(w_gate, w_up, w_down, x_bits):
    """a6: Eq. (1) over all channels -> (h[F], y[d]) in fp64."""
    lib = _load()
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    x = _c(x_bits, np.uint16).ravel()
    F, d = wg.shape
    h = np.empty(F)
    y = np.empty(d)
    _check(lib.oracle_dense_ffn(F, d, _p(wg), _p(wu), _p(wd), _p(x), _p(h), _p(y)), "dense_ffn")
    return h, y


class Proxy:
    """Quantized proxy of one layer (a0), as the oracle defines it."""

    def __init__(self, w_gate, w_up):
        self.q_gate, self.s_gate = quantize(w_gate)
        self.q_up, self.s_up = quantize(w_up)


def prox_ffn(w_gate, w_up, w_down, x_bits, keep_fraction: float,
             input_keep: float = 0.5, proxy: Proxy | None = None):
    """The two-stage step; returns a dict with kept, score, idx, h, y."""
    lib = _load()
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    x = _c(x_bits, np.uint16).ravel()
    F, d = wg.shape
    if proxy is None:
        proxy = Proxy(wg, wu)
    kx = keep_count(d, input_keep)
    k = keep_count(F, keep_fraction)
    kept = np.empty(kx, dtype=np.int32)
    score = np.empty(F)
    idx = np.empty(k, dtype=np.int32)
    h = np.empty(k)
    y = np.empty(d)
    qg, qu = _c(proxy.q_gate, np.int8), _c(proxy.q_up, np.int8)
    sg, su = _c(proxy.s_gate, np.float64), _c(proxy.s_up, np.float64)
    _check(lib.oracle_prox_ffn(F, d, _p(wg), _p(wu), _p(wd), _p(qg), _p(sg), _p(qu), _p(su),
                               _p(x), kx, k, _p(kept), _p(score), _p(idx), _p(h), _p(y)),
           "prox_ffn")
    return {"kept": kept, "score": score, "idx": idx, "h": h, "y": y, "kx": kx, "k": k}


def residual_rmsnorm(x_bits, y, eps: float = 1e-6) -> np.ndarray:
    """Stack glue: bf16(RMSNorm(x + y)) without a gain; returns bf16 bits."""
    lib = _load()
    x = _c(x_bits, np.uint16).ravel()
    yy = _c(y, np.float64).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    _check(lib.oracle_residual_rmsnorm(x.size, _p(x), _p(yy), float(eps), _p(out)),
           "residual_rmsnorm")
    return out


# ---------------------------------------------------------------- int8 Stage 2
def quantize_rows_q8(w_bits):
    """Per-row symmetric int8 of a [rows][n] bf16 matrix (reading of "compatible
    with quantization", Prox Abstract): returns (q int8 [rows][n], s float32 [rows])."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    rows, n = w.shape
    q = np.empty((rows, n), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    _check(lib.oracle_quantize_rows_q8(rows, n, _p(w), _p(q), _p(s)), "quantize_rows_q8")
    return q, s


def stage2_q8(w_gate, w_up, w_down):
    """int8 Stage-2 weights: rows of W_gate and W_up, rows of W_down^T."""
    qg, sg = quantize_rows_q8(w_gate)
    qu, su = quantize_rows_q8(w_up)
    qd, sd = quantize_rows_q8(np.ascontiguousarray(np.asarray(w_down).T))
    return {"q_gate": qg, "s_gate": sg, "q_up": qu, "s_up": su, "q_down": qd, "s_down": sd}


def quantize_rows_q4(w_bits):
    """Per-row symmetric int4 of a [rows][n] bf16 matrix (the int4 reading of
    "compatible with quantization", Prox Abstract): returns (q int8 [rows][n]
    with values in [-8, 7], s float32 [rows])."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    rows, n = w.shape
    q = np.empty((rows, n), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    _check(lib.oracle_quantize_rows_q4(rows, n, _p(w), _p(q), _p(s)), "quantize_rows_q4")
    return q, s


def stage2_q4(w_gate, w_up, w_down):
    """int4 Stage-2 weights: rows of W_gate and W_up, rows of W_down^T; the
    same dictionary as stage2_q8, so sparse_ffn_q8 evaluates Stage 2 on them."""
    qg, sg = quantize_rows_q4(w_gate)
    qu, su = quantize_rows_q4(w_up)
    qd, sd = quantize_rows_q4(np.ascontiguousarray(np.asarray(w_down).T))
    return {"q_gate": qg, "s_gate": sg, "q_up": qu, "s_up": su, "q_down": qd, "s_down": sd}


def sparse_ffn_q8(q8, x_bits, idx):
    """Stage 2 with int8 weights on the channels idx: returns (h, y) in fp64."""
    lib = _load()
    x = _c(x_bits, np.uint16).ravel()
    idx = _c(idx, np.int32).ravel()
    F, d = q8["q_gate"].shape
    h = np.empty(max(idx.size, 1), dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    arrs = [_c(q8[k], t) for k, t in (("q_gate", np.int8), ("s_gate", np.float32),
                                      ("q_up", np.int8), ("s_up", np.float32),
                                      ("q_down", np.int8), ("s_down", np.float32))]
    _check(lib.oracle_sparse_ffn_q8(F, d, *[_p(a) for a in arrs], _p(x), idx.size, _p(idx),
                                    _p(h), _p(y)), "sparse_ffn_q8")
    return h[: idx.size], y
