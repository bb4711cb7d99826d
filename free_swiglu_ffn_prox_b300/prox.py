"""Thin Python binding of libprox (include/prox.h), same entry-point names.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and streams.  There
is no fallback: if ``libprox.so`` is missing or cannot be loaded, importing
the entry points raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libprox.so")

PROX_OK = 0
PROX_ERR_INVALID_ARG = 1
PROX_ERR_UNSUPPORTED_SHAPE = 2
PROX_ERR_MISALIGNED = 3
PROX_ERR_CUDA = 4
PROX_ERR_TIMEOUT = 5
PROX_ERR_DEVICE_CHECK = 6
PROX_TRACE_EVENTS = 2
PROX_PHASE_STAMPS = 16
PHASES = ("start", "input_select", "proxy", "barrier1", "scores", "mask_known", "first_row",
          "pass_a_done", "pass_b_done", "end", "input_hist", "proxy_first_row", "proxy_loop_done",
          "scores_formed", "sel_staged", "sel_kth_found")

_lock = threading.Lock()
_lib = None


class ProxError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = int(code)
        super().__init__(f"{what}: {prox_status_string(code)} (status {code})")


class _Sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("proxy_codes", "proxy_scales", "gateup", "down_t", "workspace")]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libprox.so not found at {LIB_PATH}; build it with "
                "`python -m free_swiglu_ffn_prox_b300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        sig = {
            "prox_query_sizes": (i32, [i32, i32, ctypes.POINTER(_Sizes)]),
            "prox_prepare": (i32, [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   ctypes.POINTER(vp)]),
            "prox_query_sizes_q8": (i32, [i32, i32, ctypes.POINTER(_Sizes)]),
            "prox_prepare_q8": (i32, [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.POINTER(vp)]),
            "prox_query_sizes_q4": (i32, [i32, i32, ctypes.POINTER(_Sizes)]),
            "prox_prepare_q4": (i32, [i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.POINTER(vp)]),
            "prox_ffn": (i32, [vp, vp, f32, vp, vp]),
            "prox_ffn_ex": (i32, [vp, vp, f32, f32, vp, vp]),
            "prox_ffn_host": (i32, [vp, vp, f32, vp, vp]),
            "prox_ffn_traced": (i32, [vp, vp, f32, f32, vp, ctypes.POINTER(vp), i32, vp]),
            "prox_dense_ffn": (i32, [vp, vp, vp, vp]),
            "prox_ffn_debug": (i32, [vp, vp, f32, f32, vp, vp, vp, vp, vp, vp]),
            "prox_ffn_blocks": (i32, [vp, vp, i32, f32, vp, vp]),
            "prox_ffn_batch": (i32, [vp, vp, i32, f32, vp, vp]),
            "prox_ffn_batch_union": (i32, [vp, vp, i32, f32, vp, vp]),
            "prox_ffn_batch_union_debug": (i32, [vp, vp, i32, f32, vp, vp, vp]),
            "prox_batch_union_group": (i32, [vp]),
            "prox_ffn_blocks_debug": (i32, [vp, vp, i32, f32, vp, vp, vp, vp, vp]),
            "prox_ffn_contrib": (i32, [vp, vp, f32, vp, vp]),
            "prox_stack_ffn": (i32, [ctypes.POINTER(vp), i32, vp, f32, f32, vp, vp, vp]),
            "prox_ffn_contrib_debug": (i32, [vp, vp, f32, vp, vp, vp, vp, vp]),
            "prox_residual_rmsnorm": (i32, [i32, vp, vp, f32, vp, vp]),
            "prox_ffn_resnorm": (i32, [vp, vp, vp, f32, vp, f32, vp, vp]),
            "prox_get_status": (i32, [vp, vp]),
            "prox_test_barrier_timeout": (i32, [vp, vp, vp, vp]),
            "prox_layer_blocks": (i32, [vp]),
            "prox_ffn_phase_times": (i32, [vp, vp, f32, vp, vp, i32, vp]),
            "prox_layer_info": (i32, [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "prox_keep_count": (i32, [i32, f32]),
            "prox_destroy": (None, [vp]),
            "prox_status_string": (ctypes.c_char_p, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def loaded_library_path() -> str:
    _load()
    return LIB_PATH


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(code: int, what: str) -> None:
    if code != PROX_OK:
        raise ProxError(code, what)


def _need(t: torch.Tensor, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------- entry points
def prox_status_string(code: int) -> str:
    return _load().prox_status_string(int(code)).decode()


def prox_keep_count(n: int, frac: float) -> int:
    return int(_load().prox_keep_count(int(n), float(frac)))


_PREPARE_SUFFIX = {0: "", 1: "_q8", 2: "_q4"}


def prox_query_sizes(d_model: int, d_ff: int, q8: bool = False, q4: bool = False) -> dict:
    """Buffer sizes for prox_prepare (q8: for prox_prepare_q8, q4: for
    prox_prepare_q4)."""
    if q8 and q4:
        raise ValueError("q8 and q4 are exclusive")
    s = _Sizes()
    name = "prox_query_sizes" + _PREPARE_SUFFIX[2 if q4 else 1 if q8 else 0]
    _check(getattr(_load(), name)(int(d_model), int(d_ff), ctypes.byref(s)), name)
    return {n: int(getattr(s, n)) for n, _ in _Sizes._fields_}


class ProxLayer:
    """A prepared layer: the device buffers (owned here, as torch tensors)
    and the library's host handle."""

    def __init__(self, d_model, d_ff, bufs, handle, device, wq=0):
        self.d_model, self.d_ff = int(d_model), int(d_ff)
        self.wq = int(wq)  # Stage-2 rows: 0 bf16, 1 int8, 2 int4
        self.q8 = self.wq == 1
        self.q4 = self.wq == 2
        self.bufs = bufs
        self.handle = handle
        self.device = device

    def close(self):
        if self.handle is not None and _lib is not None:
            _lib.prox_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _prepare(w_gate, w_up, w_down, stream, wq):
    lib = _load()
    if w_gate.dim() != 2:
        raise ValueError("w_gate must be [d_ff, d_model]")
    d_ff, d_model = w_gate.shape
    for t, shp, nm in ((w_gate, (d_ff, d_model), "w_gate"), (w_up, (d_ff, d_model), "w_up"),
                       (w_down, (d_model, d_ff), "w_down")):
        _need(t, torch.bfloat16, shp, nm)
    sz = prox_query_sizes(d_model, d_ff, q8=wq == 1, q4=wq == 2)
    dev = w_gate.device
    bufs = {n: torch.empty(sz[n], dtype=torch.uint8, device=dev) for n in sz}
    h = ctypes.c_void_p()
    name = "prox_prepare" + _PREPARE_SUFFIX[wq]
    with torch.cuda.device(dev):
        _check(getattr(lib, name)(d_model, d_ff, _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                  _ptr(bufs["proxy_codes"]), _ptr(bufs["proxy_scales"]),
                                  _ptr(bufs["gateup"]), _ptr(bufs["down_t"]),
                                  _ptr(bufs["workspace"]), _stream(stream), ctypes.byref(h)),
               name)
    return ProxLayer(d_model, d_ff, bufs, h, dev, wq)


def prox_prepare(w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                 stream=None) -> ProxLayer:
    """Builds the proxy and Stage-2 layouts of one layer (see prox.h)."""
    return _prepare(w_gate, w_up, w_down, stream, 0)


def prox_prepare_q8(w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                    stream=None) -> ProxLayer:
    """As prox_prepare with int8 Stage-2 rows (see prox.h); every step call on
    the returned layer runs Stage 2 on them.  bufs["gateup"] and
    bufs["down_t"] hold the int8 layouts."""
    return _prepare(w_gate, w_up, w_down, stream, 1)


def prox_prepare_q4(w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                    stream=None) -> ProxLayer:
    """As prox_prepare with int4 Stage-2 rows (see prox.h); bufs["gateup"]
    and bufs["down_t"] hold the int4 layouts."""
    return _prepare(w_gate, w_up, w_down, stream, 2)


def _x_y(layer: ProxLayer, x, y):
    _need(x, torch.bfloat16, (layer.d_model,), "x")
    if y is None:
        y = torch.empty(layer.d_model, dtype=torch.float32, device=x.device)
    _need(y, torch.float32, (layer.d_model,), "y")
    return y


def prox_ffn(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, y=None, stream=None):
    y = _x_y(layer, x, y)
    _check(_load().prox_ffn(layer.handle, _ptr(x), float(keep_fraction), _ptr(y), _stream(stream)),
           "prox_ffn")
    return y


def prox_ffn_ex(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, input_keep: float,
                y=None, stream=None):
    y = _x_y(layer, x, y)
    _check(_load().prox_ffn_ex(layer.handle, _ptr(x), float(keep_fraction), float(input_keep),
                               _ptr(y), _stream(stream)), "prox_ffn_ex")
    return y


def prox_ffn_host(layer: ProxLayer, x_host: torch.Tensor, keep_fraction: float, y_host=None,
                  stream=None):
    """prox_ffn on host tensors: the library copies x in and y out on the
    stream.  Pinned tensors give asynchronous copies; y_host is valid once
    the stream has passed the call."""
    if not isinstance(x_host, torch.Tensor) or x_host.is_cuda:
        raise ValueError("x_host must be a host tensor")
    if x_host.dtype != torch.bfloat16 or tuple(x_host.shape) != (layer.d_model,) \
            or not x_host.is_contiguous():
        raise ValueError(f"x_host must be a contiguous bf16 tensor of shape ({layer.d_model},)")
    if y_host is None:
        y_host = torch.empty(layer.d_model, dtype=torch.float32, pin_memory=x_host.is_pinned())
    if y_host.is_cuda or y_host.dtype != torch.float32 or tuple(y_host.shape) != (layer.d_model,) \
            or not y_host.is_contiguous():
        raise ValueError(f"y_host must be a contiguous fp32 host tensor of shape ({layer.d_model},)")
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_host(layer.handle, _ptr(x_host), float(keep_fraction),
                                     _ptr(y_host), _stream(stream)), "prox_ffn_host")
    return y_host


def prox_ffn_traced(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, events,
                    input_keep: float = 0.5, y=None, stream=None):
    """prox_ffn_ex recording ``events`` (PROX_TRACE_EVENTS timing-enabled
    torch.cuda.Event objects, each already recorded once so that it exists)
    around its kernel; events[0].elapsed_time(events[1]) is the step."""
    y = _x_y(layer, x, y)
    if len(events) != PROX_TRACE_EVENTS:
        raise ValueError(f"need {PROX_TRACE_EVENTS} events")
    handles = (ctypes.c_void_p * PROX_TRACE_EVENTS)(*[int(e.cuda_event) for e in events])
    _check(_load().prox_ffn_traced(layer.handle, _ptr(x), float(keep_fraction), float(input_keep),
                                   _ptr(y), handles, PROX_TRACE_EVENTS, _stream(stream)),
           "prox_ffn_traced")
    return y


def prox_ffn_noalloc(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, y=None,
                     stream=None):
    """prox_ffn whose per-step scratch lives in a fixed array inside the
    library (no workspace of the caller's is used).  For callers that cannot
    allocate device memory while stepping; see prox.h for the limits (the
    layer's workspace must fit in 4 MiB; overlapping calls race)."""
    lib = _load()
    fn = lib.prox_ffn_noalloc
    if fn.argtypes is None:
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                       ctypes.c_void_p]
    y = _x_y(layer, x, y)
    _check(fn(layer.handle, _ptr(x), float(keep_fraction), _ptr(y), _stream(stream)),
           "prox_ffn_noalloc")
    return y


def prox_ffn_contrib(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, y=None,
                     stream=None):
    """The decode step ranking channels by |h~_c| ||W_down[:, c]|| (the
    COUNTDOWN-style contribution signal) instead of |h~_c|."""
    y = _x_y(layer, x, y)
    _check(_load().prox_ffn_contrib(layer.handle, _ptr(x), float(keep_fraction), _ptr(y),
                                    _stream(stream)), "prox_ffn_contrib")
    return y


def prox_ffn_contrib_debug(layer: ProxLayer, x: torch.Tensor, keep_fraction: float,
                           stream=None) -> dict:
    """prox_ffn_contrib plus its scores, channel list and h (device tensors)."""
    y = _x_y(layer, x, None)
    dev = x.device
    k = prox_keep_count(layer.d_ff, keep_fraction)
    scores = torch.empty(layer.d_ff, dtype=torch.float32, device=dev)
    idx = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
    h = torch.empty(max(k, 1), dtype=torch.float32, device=dev)
    _check(_load().prox_ffn_contrib_debug(layer.handle, _ptr(x), float(keep_fraction), _ptr(y),
                                          _ptr(scores), _ptr(idx), _ptr(h), _stream(stream)),
           "prox_ffn_contrib_debug")
    return {"y": y, "scores": scores, "idx": idx[:k], "h": h[:k], "k": k}


def prox_stack_ffn(layers, x0: torch.Tensor, keep_fraction: float, eps: float = 1e-6,
                   xs=None, ys=None, stream=None):
    """n layers in one persistent launch: layer 0 on x0, layer l > 0 on
    x_l = bf16(RMSNorm(x_{l-1} + y_{l-1})).  Returns (xs bf16 [n][d] with row l
    = x_l for l >= 1, ys fp32 [n][d] with row l = y_l)."""
    n = len(layers)
    d = layers[0].d_model
    _need(x0, torch.bfloat16, (d,), "x0")
    if xs is None:
        xs = torch.zeros(n, d, dtype=torch.bfloat16, device=x0.device)
    if ys is None:
        ys = torch.empty(n, d, dtype=torch.float32, device=x0.device)
    _need(xs, torch.bfloat16, (n, d), "xs")
    _need(ys, torch.float32, (n, d), "ys")
    handles = (ctypes.c_void_p * n)(*[L.handle.value if isinstance(L.handle, ctypes.c_void_p)
                                      else L.handle for L in layers])
    _check(_load().prox_stack_ffn(ctypes.cast(handles, ctypes.POINTER(ctypes.c_void_p)), n,
                                  _ptr(x0), float(keep_fraction), float(eps), _ptr(xs), _ptr(ys),
                                  _stream(stream)), "prox_stack_ffn")
    return xs, ys


def prox_dense_ffn(layer: ProxLayer, x: torch.Tensor, y=None, stream=None):
    y = _x_y(layer, x, y)
    _check(_load().prox_dense_ffn(layer.handle, _ptr(x), _ptr(y), _stream(stream)),
           "prox_dense_ffn")
    return y


def prox_ffn_debug(layer: ProxLayer, x: torch.Tensor, keep_fraction: float,
                   input_keep: float = 0.5, stream=None) -> dict:
    """prox_ffn_ex plus kept inputs, scores, channel list and h (device tensors)."""
    y = _x_y(layer, x, None)
    dev = x.device
    kx = prox_keep_count(layer.d_model, input_keep)
    k = prox_keep_count(layer.d_ff, keep_fraction)
    kept = torch.empty(max(kx, 1), dtype=torch.int32, device=dev)
    scores = torch.empty(layer.d_ff, dtype=torch.float32, device=dev)
    idx = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
    h = torch.empty(max(k, 1), dtype=torch.float32, device=dev)
    _check(_load().prox_ffn_debug(layer.handle, _ptr(x), float(keep_fraction), float(input_keep),
                                  _ptr(y), _ptr(kept), _ptr(scores), _ptr(idx), _ptr(h),
                                  _stream(stream)), "prox_ffn_debug")
    return {"y": y, "kept": kept[:kx], "scores": scores, "idx": idx[:k], "h": h[:k],
            "kx": kx, "k": k}


def prox_ffn_batch(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, y=None,
                   stream=None):
    """Per-token Prox steps over a batch: x bf16 [B, d_model] -> y fp32 [B, d_model]."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [batch, d_model] tensor")
    B = x.shape[0]
    _need(x, torch.bfloat16, (B, layer.d_model), "x")
    if y is None:
        y = torch.empty(B, layer.d_model, dtype=torch.float32, device=x.device)
    _need(y, torch.float32, (B, layer.d_model), "y")
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_batch(layer.handle, _ptr(x), int(B), float(keep_fraction),
                                      _ptr(y), _stream(stream)), "prox_ffn_batch")
    return y


def _batch_x_y(layer, x, y):
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [batch, d_model] tensor")
    B = x.shape[0]
    _need(x, torch.bfloat16, (B, layer.d_model), "x")
    if y is None:
        y = torch.empty(B, layer.d_model, dtype=torch.float32, device=x.device)
    _need(y, torch.float32, (B, layer.d_model), "y")
    return B, y


def prox_batch_union_group(layer: ProxLayer) -> int:
    """Tokens per pass of prox_ffn_batch_union on this layer (0: unsupported)."""
    return int(_load().prox_batch_union_group(layer.handle))


def prox_ffn_batch_union(layer: ProxLayer, x: torch.Tensor, keep_fraction: float, y=None,
                         stream=None):
    """Per-token masks, Stage 2 over their union: x bf16 [B, d_model] -> y fp32
    [B, d_model]; each row in the union is read once for the whole pass."""
    B, y = _batch_x_y(layer, x, y)
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_batch_union(layer.handle, _ptr(x), int(B), float(keep_fraction),
                                            _ptr(y), _stream(stream)), "prox_ffn_batch_union")
    return y


def prox_ffn_batch_union_debug(layer: ProxLayer, x: torch.Tensor, keep_fraction: float,
                               stream=None) -> dict:
    """prox_ffn_batch_union plus the per-channel token bits (batch <= one pass):
    {"y": [B, d_model] fp32, "member": [d_ff] int64 bit words, "masks": list
    of each token's selected channels (ascending int64 tensors)}."""
    B, y = _batch_x_y(layer, x, None)
    member = torch.zeros(layer.d_ff + 4, dtype=torch.int32, device=x.device)
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_batch_union_debug(layer.handle, _ptr(x), int(B),
                                                  float(keep_fraction), _ptr(y), _ptr(member),
                                                  _stream(stream)), "prox_ffn_batch_union_debug")
    m = member[: layer.d_ff].to(torch.int64) & 0xFFFFFFFF
    masks = [torch.nonzero((m >> t) & 1).flatten() for t in range(B)]
    return {"y": y, "member": m, "masks": masks}


def prox_ffn_blocks(layer: ProxLayer, x: torch.Tensor, block_width: int, keep_fraction: float,
                    y=None, stream=None):
    """The step with a block-granular mask: the ceil(keep_fraction E) blocks
    of block_width contiguous channels with the largest summed proxy score."""
    y = _x_y(layer, x, y)
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_blocks(layer.handle, _ptr(x), int(block_width),
                                       float(keep_fraction), _ptr(y), _stream(stream)),
               "prox_ffn_blocks")
    return y


def prox_ffn_blocks_debug(layer: ProxLayer, x: torch.Tensor, block_width: int,
                          keep_fraction: float, stream=None) -> dict:
    """prox_ffn_blocks plus per-channel scores, the channel list and h."""
    y = _x_y(layer, x, None)
    dev = x.device
    E = layer.d_ff // int(block_width) if block_width > 0 else 0
    k = int(block_width) * prox_keep_count(E, keep_fraction) if E > 0 else 0
    scores = torch.empty(layer.d_ff, dtype=torch.float32, device=dev)
    idx = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
    h = torch.empty(max(k, 1), dtype=torch.float32, device=dev)
    with torch.cuda.device(layer.device):
        _check(_load().prox_ffn_blocks_debug(layer.handle, _ptr(x), int(block_width),
                                             float(keep_fraction), _ptr(y), _ptr(scores),
                                             _ptr(idx), _ptr(h), _stream(stream)),
               "prox_ffn_blocks_debug")
    return {"y": y, "scores": scores, "idx": idx[:k], "h": h[:k], "k": k}


def prox_residual_rmsnorm(x: torch.Tensor, y: torch.Tensor, eps: float = 1e-6, out=None,
                          stream=None):
    d = x.numel()
    _need(x, torch.bfloat16, (d,), "x")
    _need(y, torch.float32, (d,), "y")
    if out is None:
        out = torch.empty(d, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (d,), "out")
    _check(_load().prox_residual_rmsnorm(d, _ptr(x), _ptr(y), float(eps), _ptr(out),
                                         _stream(stream)), "prox_residual_rmsnorm")
    return out


def prox_ffn_resnorm(layer: ProxLayer, x_prev: torch.Tensor, y_prev: torch.Tensor,
                     keep_fraction: float, eps: float = 1e-6, x_out=None, y=None, stream=None):
    """One stacked layer with the residual + RMSNorm glue fused into the step:
    x = bf16(RMSNorm(x_prev + y_prev)) (written to x_out), y = the step on x.
    Returns (x_out, y)."""
    d = layer.d_model
    _need(x_prev, torch.bfloat16, (d,), "x_prev")
    _need(y_prev, torch.float32, (d,), "y_prev")
    if x_out is None:
        x_out = torch.empty(d, dtype=torch.bfloat16, device=x_prev.device)
    if y is None:
        y = torch.empty(d, dtype=torch.float32, device=x_prev.device)
    _need(x_out, torch.bfloat16, (d,), "x_out")
    _need(y, torch.float32, (d,), "y")
    _check(_load().prox_ffn_resnorm(layer.handle, _ptr(x_prev), _ptr(y_prev), float(eps),
                                    _ptr(x_out), float(keep_fraction), _ptr(y), _stream(stream)),
           "prox_ffn_resnorm")
    return x_out, y


def prox_get_status(layer: ProxLayer, stream=None) -> int:
    return int(_load().prox_get_status(layer.handle, _stream(stream)))


def prox_layer_blocks(layer: ProxLayer) -> int:
    return int(_load().prox_layer_blocks(layer.handle))


def prox_ffn_phase_times(layer: ProxLayer, x: torch.Tensor, keep_fraction: float = 0.3,
                         dense: bool = False, stream=None):
    """One step with per-CTA %globaltimer stamps at the phase boundaries;
    returns (y, stamps int64 [blocks][PROX_PHASE_STAMPS] on the device)."""
    y = _x_y(layer, x, None)
    nb = prox_layer_blocks(layer)
    ts = torch.zeros(nb, PROX_PHASE_STAMPS, dtype=torch.int64, device=x.device)
    _check(_load().prox_ffn_phase_times(layer.handle, _ptr(x), float(keep_fraction), _ptr(y),
                                        _ptr(ts), int(bool(dense)), _stream(stream)),
           "prox_ffn_phase_times")
    return y, ts


def prox_test_barrier_timeout(layer: ProxLayer, x: torch.Tensor, stream=None) -> int:
    """Failure-detection test hook: a step whose first grid barrier can not
    complete; returns the status the bounded waits recorded."""
    y = _x_y(layer, x, None)
    return int(_load().prox_test_barrier_timeout(layer.handle, _ptr(x), _ptr(y), _stream(stream)))


def prox_layer_info(layer: ProxLayer):
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(_load().prox_layer_info(layer.handle, ctypes.byref(a), ctypes.byref(b)), "prox_layer_info")
    return a.value, b.value


def prox_destroy(layer: ProxLayer) -> None:
    layer.close()
