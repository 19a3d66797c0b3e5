"""Gated delta rule on GB300 (sm_103a): Python binding of libgdn.so.

The functions here only marshal arguments: every step of the computation
runs in the CUDA kernels behind the C ABI declared in ``include/gdn.h``.
There is no CPU or PyTorch fallback; if the library is not built, every
call raises.

Low level (same names and argument order as the C ABI; torch tensors in,
raise ``GdnError`` on a non-zero status):
    gdn_prefill(q, k, v, g, beta, state_in, state_out, y, chunk, workspace=None, stream=None)
    gdn_decode_step(q, k, v, g, beta, state_in, state_out, y, stream=None)
    gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, dtype)
    gdn_status_string(status)
Convenience (allocates the outputs with torch):
    prefill(q, k, v, g, beta, state_in=None, chunk=64) -> (y, state_out)
    decode_step(q, k, v, g, beta, state) -> y        (state updated in place)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_ALIGNMENT = -3
GDN_ERR_WORKSPACE = -4
GDN_ERR_CUDA = -5
GDN_ERR_DEVICE_TIMEOUT = -6
GDN_ERR_NOALLOC_LIMIT = -7
GDN_NOALLOC_SCRATCH_BYTES = 32 << 20
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1
GDN_DTYPE_F16 = 2
GDN_OPT_TILED_HEADS = 1
GDN_OPT_LOG_GATE = 2
GDN_OPT_L2NORM_QK = 4

_DTYPES = {torch.float32: GDN_DTYPE_F32, torch.bfloat16: GDN_DTYPE_BF16,
           torch.float16: GDN_DTYPE_F16}
_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({gdn_status_string(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m gated_delta_rule_02_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.gdn_prefill_workspace_bytes.argtypes = [i] * 8
            L.gdn_prefill_workspace_bytes.restype = sz
            L.gdn_prefill.argtypes = [vp] * 8 + [i] * 8 + [vp, sz, vp]
            L.gdn_prefill.restype = i
            L.gdn_decode_step.argtypes = [vp] * 8 + [i] * 6 + [vp]
            L.gdn_decode_step.restype = i
            L.gdn_status_string.argtypes = [i]
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_device_status.argtypes = [i]
            L.gdn_device_status.restype = i
            L.gdn_prefill_noalloc.argtypes = [vp] * 8 + [i] * 8 + [vp]
            L.gdn_prefill_noalloc.restype = i
            L.gdn_prefill_ex.argtypes = [vp] * 8 + [i] * 8 + [vp, sz, vp, i]
            L.gdn_prefill_ex.restype = i
            L.gdn_decode_step_ex.argtypes = [vp] * 8 + [i] * 6 + [vp, i]
            L.gdn_decode_step_ex.restype = i
            L.gdn_selftest_wait_timeout.argtypes = [vp]
            L.gdn_selftest_wait_timeout.restype = i
            _lib = L
    return _lib


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def gdn_device_status(clear: bool = False) -> int:
    """GDN_OK, or GDN_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up
    (synchronises the device)."""
    return int(lib().gdn_device_status(1 if clear else 0))


def gdn_selftest_wait_timeout(stream=None, device=None) -> None:
    """Enqueue ``gdn_selftest_wait_timeout`` (include/gdn.h): a kernel whose
    bounded waits run out (about 4 s), so that the next ``gdn_device_status``
    reports GDN_ERR_DEVICE_TIMEOUT."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    st = lib().gdn_selftest_wait_timeout(_stream_handle(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_selftest_wait_timeout")


def gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, dtype) -> int:
    if isinstance(dtype, torch.dtype):
        dtype = _DTYPES[dtype]
    return int(lib().gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, dtype))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(tensors, dtype, device):
    for name, t in tensors:
        if t is None:
            continue
        if not t.is_cuda or t.device != device:
            raise ValueError(f"{name} must be a CUDA tensor on {device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def gdn_prefill(q, k, v, g, beta, state_in, state_out, y, chunk, workspace=None,
                stream=None, options=0):
    """Enqueue ``gdn_prefill`` (include/gdn.h) on ``stream`` (default: current);
    with ``options`` (GDN_OPT_* bits) ``gdn_prefill_ex``."""
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    dev = q.device
    _check([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("y", y)], dt, dev)
    _check([("state_in", state_in), ("state_out", state_out)], torch.float32, dev)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    need = gdn_prefill_workspace_bytes(B, T, Hk, Hv, Dk, Dv, chunk, _DTYPES[dt])
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(state_out),
            _ptr(y), B, T, Hk, Hv, Dk, Dv, int(chunk), _DTYPES[dt], _ptr(workspace), ws_bytes,
            _stream_handle(stream, dev))
    if options:
        st = lib().gdn_prefill_ex(*args, int(options))
    else:
        st = lib().gdn_prefill(*args)
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill_ex" if options else "gdn_prefill")


def gdn_prefill_noalloc(q, k, v, g, beta, state_in, state_out, y, chunk, stream=None):
    """Enqueue ``gdn_prefill_noalloc`` (include/gdn.h): the prefill without a
    caller workspace, using the library's fixed scratch buffer instead."""
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    dev = q.device
    _check([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("y", y)], dt, dev)
    _check([("state_in", state_in), ("state_out", state_out)], torch.float32, dev)
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    st = lib().gdn_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(state_in), _ptr(state_out), _ptr(y),
                                   B, T, Hk, Hv, Dk, Dv, int(chunk), _DTYPES[dt],
                                   _stream_handle(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill_noalloc")


def gdn_decode_step(q, k, v, g, beta, state_in, state_out, y, stream=None, options=0):
    """Enqueue ``gdn_decode_step`` (include/gdn.h) on ``stream`` (default: current);
    with ``options`` (GDN_OPT_* bits) ``gdn_decode_step_ex``."""
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    dev = q.device
    _check([("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("y", y)], dt, dev)
    _check([("state_in", state_in), ("state_out", state_out)], torch.float32, dev)
    B, _, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(state_out),
            _ptr(y), B, Hk, Hv, Dk, Dv, _DTYPES[dt], _stream_handle(stream, dev))
    if options:
        st = lib().gdn_decode_step_ex(*args, int(options))
    else:
        st = lib().gdn_decode_step(*args)
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_step_ex" if options else "gdn_decode_step")


def prefill(q, k, v, g, beta, state_in=None, chunk=64, stream=None, options=0):
    """Run the prefill; returns ``(y, state_out)`` (new tensors)."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    y = torch.empty((B, T, Hv, Dv), dtype=q.dtype, device=q.device)
    state_out = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=q.device)
    gdn_prefill(q, k, v, g, beta, state_in, state_out, y, chunk, stream=stream, options=options)
    return y, state_out


def decode_step(q, k, v, g, beta, state, stream=None, options=0):
    """One decode step; ``state`` is updated in place, returns ``y``."""
    B = q.shape[0]
    Hv, Dv = v.shape[2], v.shape[3]
    y = torch.empty((B, 1, Hv, Dv), dtype=q.dtype, device=q.device)
    gdn_decode_step(q, k, v, g, beta, state, state, y, stream=stream, options=options)
    return y
