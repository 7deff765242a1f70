"""Thin ctypes binding of ``libpalimpsa.so`` (declared in ``include/palimpsa.h``).

The functions keep the C names. They only marshal arguments: shapes and dtypes
are read from torch tensors, device pointers and the current CUDA stream are
passed through, and a non-OK status raises :class:`PalimpsaError`. Every step
of the computation runs in the library's CUDA kernels; there is no fallback,
and a missing library raises instead of computing anything another way.

Host (CPU) tensors are accepted too: they are copied to the current CUDA
device, the kernels run there, and the results are copied back before the call
returns (the end-to-end path a caller with host buffers uses).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build_lib

PALIMPSA_F32 = 0
PALIMPSA_BF16 = 1
STATUS_NAMES = {
    0: "PALIMPSA_OK", 1: "PALIMPSA_ERR_NULL", 2: "PALIMPSA_ERR_SHAPE", 3: "PALIMPSA_ERR_ALIGN",
    4: "PALIMPSA_ERR_DTYPE", 5: "PALIMPSA_ERR_DOMAIN", 6: "PALIMPSA_ERR_UNSUPPORTED",
    7: "PALIMPSA_ERR_CUDA", 8: "PALIMPSA_ERR_TIMEOUT", 9: "PALIMPSA_ERR_SCRATCH_LIMIT",
}

_lib = None
_lock = threading.Lock()


class PalimpsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = palimpsa_status_string(code) if _lib is not None else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(self.code, self.code)} ({msg})")


def library_path() -> str:
    return build_lib.LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of libpalimpsa.so."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or build_lib.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -m metaplastic_linear_attention_gb300.build_lib)")
        lib = ctypes.CDLL(path)
        vp, fp, i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
        lib.palimpsa_forward_chunked.restype = i
        lib.palimpsa_forward_chunked.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp,
                                                 i, i, i, i, i, i, i, vp]
        lib.palimpsa_forward_chunked_noalloc.restype = i
        lib.palimpsa_forward_chunked_noalloc.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp,
                                                         i, i, i, i, i, i, i, vp]
        lib.palimpsa_step.restype = i
        lib.palimpsa_step.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, vp]
        lib.palimpsa_status_string.restype = ctypes.c_char_p
        lib.palimpsa_status_string.argtypes = [i]
        lib.palimpsa_get_device_status.restype = i
        lib.palimpsa_get_device_status.argtypes = [vp]
        lib.palimpsa_abi_version.restype = i
        lib.palimpsa_abi_version.argtypes = []
        lib.palimpsa_set_wait_timeout_ns.restype = None
        lib.palimpsa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.palimpsa_debug_withhold_first_copy.restype = None
        lib.palimpsa_debug_withhold_first_copy.argtypes = [i]
        lib.palimpsa_set_forward_segments.restype = None
        lib.palimpsa_set_forward_segments.argtypes = [i]
        _lib = lib
        return lib


def palimpsa_status_string(code: int) -> str:
    return load_library().palimpsa_status_string(int(code)).decode()


def palimpsa_abi_version() -> int:
    return int(load_library().palimpsa_abi_version())


def palimpsa_set_wait_timeout_ns(ns: int) -> None:
    load_library().palimpsa_set_wait_timeout_ns(int(ns))


def palimpsa_debug_withhold_first_copy(on: bool) -> None:
    load_library().palimpsa_debug_withhold_first_copy(1 if on else 0)


def palimpsa_set_forward_segments(segments: int) -> None:
    load_library().palimpsa_set_forward_segments(int(segments))


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def palimpsa_get_device_status(stream=None) -> int:
    """Synchronise the stream, read and clear the device status word (returns the code)."""
    return int(load_library().palimpsa_get_device_status(ctypes.c_void_p(_stream_handle(stream))))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _in_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PALIMPSA_BF16
    if t.dtype == torch.float32:
        return PALIMPSA_F32
    raise TypeError(f"q, k, v, beta must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, shape, dtype=None, device=None):
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _to_device(ts, device):
    return [None if t is None else t.to(device, non_blocking=True) for t in ts]


def _compute_device(*ts):
    """The CUDA device of the first CUDA tensor among ts, else the current device."""
    for t in ts:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _deliver(dst, src):
    """Return src in the caller's placement: dst itself when it is the device
    result, a host copy into dst, or a new pinned host tensor when dst is None."""
    if dst is not None and dst.is_cuda:
        return dst
    if dst is None:
        dst = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
    dst.copy_(src, non_blocking=True)
    return dst


def palimpsa_forward_chunked(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None, *, y=None, mu_T=None,
                             I_T=None, chunk: int = 0, stream=None):
    """Recurrence over T tokens (see palimpsa.h). Returns (y, mu_T, I_T).

    q, k [B,H,T,d_k] and v, beta [B,H,T,d_v] share one dtype (bf16 or fp32);
    d_t [B,H,T], A [H], I_prior [H], mu0/I0 [B,H,d_v,d_k] are fp32. Outputs are
    allocated when not given; mu_T / I_T may be mu0 / I0 (in place).
    """
    if q.device.type == "cpu":
        # Host inputs: copy them in, compute on the device, and deliver each output
        # where the caller's tensor lives (a host output is copied back; a CUDA
        # output, e.g. a resident decode state, is written in place).
        dev = _compute_device(y, mu_T, I_T, mu0, I0)
        dq = _to_device([q, k, v, beta, d_t, A, I_prior, mu0, I0], dev)
        dev_out = [o if (o is not None and o.is_cuda) else None for o in (y, mu_T, I_T)]
        res = palimpsa_forward_chunked(*dq, y=dev_out[0], mu_T=dev_out[1], I_T=dev_out[2], chunk=chunk,
                                       stream=stream)
        outs = [_deliver(dst, src) for dst, src in zip((y, mu_T, I_T), res)]
        (stream or torch.cuda.current_stream()).synchronize()
        return tuple(outs)

    B, H, T, d_k = q.shape
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    _check(k, "k", q.shape, q.dtype, dev)
    _check(v, "v", (B, H, T, d_v), q.dtype, dev)
    _check(beta, "beta", (B, H, T, d_v), q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(d_t, "d_t", (B, H, T), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(mu0, "mu0", (B, H, d_v, d_k), f32, dev)
    _check(I0, "I0", (B, H, d_v, d_k), f32, dev)
    if y is None:
        y = torch.empty((B, H, T, d_v), dtype=f32, device=dev)
    if mu_T is None:
        mu_T = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev)
    if I_T is None:
        I_T = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev)
    _check(y, "y", (B, H, T, d_v), f32, dev)
    _check(mu_T, "mu_T", (B, H, d_v, d_k), f32, dev)
    _check(I_T, "I_T", (B, H, d_v, d_k), f32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_forward_chunked(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(I0),
            _ptr(y), _ptr(mu_T), _ptr(I_T), B, H, T, d_k, d_v, int(chunk), _in_dtype(q),
            ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_chunked")
    return y, mu_T, I_T


def palimpsa_step(q, k, v, beta, d_t, A, I_prior, mu, I, *, y=None, stream=None):
    """One decode token (see palimpsa.h): updates mu, I in place and returns y [B,H,d_v]."""
    if q.device.type == "cpu":
        # Host inputs: the state stays where it is when it is on the device (the
        # resident decode state); host state is copied in and back.
        dev = _compute_device(mu, I, y)
        dq = _to_device([q, k, v, beta, d_t, A, I_prior, mu, I], dev)
        ydev = y if (y is not None and y.is_cuda) else None
        ry = palimpsa_step(*dq, y=ydev, stream=stream)
        if not mu.is_cuda:
            mu.copy_(dq[7], non_blocking=True)
        if not I.is_cuda:
            I.copy_(dq[8], non_blocking=True)
        out = _deliver(y, ry)
        (stream or torch.cuda.current_stream()).synchronize()
        return out

    B, H, d_k = q.shape
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    _check(k, "k", q.shape, q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(v, "v", (B, H, d_v), q.dtype, dev)
    _check(beta, "beta", (B, H, d_v), q.dtype, dev)
    _check(d_t, "d_t", (B, H), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(mu, "mu", (B, H, d_v, d_k), f32, dev)
    _check(I, "I", (B, H, d_v, d_k), f32, dev)
    if y is None:
        y = torch.empty((B, H, d_v), dtype=f32, device=dev)
    _check(y, "y", (B, H, d_v), f32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior),
                               _ptr(mu), _ptr(I), _ptr(y), B, H, d_k, d_v, _in_dtype(q),
                               ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_step")
    return y
