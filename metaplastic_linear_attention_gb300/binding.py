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
PALIMPSA_FUSE_QK_NORM = 1   # palimpsa_fuse_flags
PALIMPSA_FUSE_V_STAR = 2
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
        lib.palimpsa_forward_without_meta.restype = i
        lib.palimpsa_forward_without_meta.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp,
                                                      i, i, i, i, i, i, i, vp]
        lib.palimpsa_backward.restype = i
        lib.palimpsa_backward.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                          fp, fp, fp, i, i, i, i, i, i, vp]
        u = ctypes.c_uint
        lib.palimpsa_forward_fused.restype = i
        lib.palimpsa_forward_fused.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                               i, i, i, i, i, i, u, i, vp]
        lib.palimpsa_forward_varlen_fused.restype = i
        lib.palimpsa_forward_varlen_fused.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp, vp,
                                                      i, i, i, i, i, i, i, ctypes.c_uint, i, vp]
        lib.palimpsa_forward_varlen.restype = i
        lib.palimpsa_forward_varlen.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, vp,
                                                i, i, i, i, i, i, i, i, vp]
        lib.palimpsa_segment_summary.restype = i
        lib.palimpsa_segment_summary.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, i, i, i, i, i, i, i, vp]
        lib.palimpsa_state_combine.restype = i
        lib.palimpsa_state_combine.argtypes = [fp, fp, i, fp, fp, fp, fp, fp, i, i, i, i, vp]
        lib.palimpsa_checkpoint_bytes.restype = ctypes.c_size_t
        lib.palimpsa_checkpoint_bytes.argtypes = [i, i, i, i, i]
        lib.palimpsa_forward_checkpointed.restype = i
        lib.palimpsa_forward_checkpointed.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                                      i, i, i, i, i, i, i, vp]
        lib.palimpsa_backward_checkpointed.restype = i
        lib.palimpsa_backward_checkpointed.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                                       fp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp]
        lib.palimpsa_checkpoint_bytes_varlen.restype = ctypes.c_size_t
        lib.palimpsa_checkpoint_bytes_varlen.argtypes = [i, i, i, i, i]
        lib.palimpsa_forward_varlen_checkpointed.restype = i
        lib.palimpsa_forward_varlen_checkpointed.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp, vp,
                                                             i, i, i, i, i, i, i, i, vp]
        lib.palimpsa_backward_varlen.restype = i
        lib.palimpsa_backward_varlen.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp, fp,
                                                 fp, fp, fp, fp, fp, vp, i, i, i, i, i, i, i, vp]
        lib.palimpsa_forward_plan.restype = i
        lib.palimpsa_forward_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_size_t)]
        lib.palimpsa_step_fused.restype = i
        lib.palimpsa_step_fused.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, i, i, i, i, u, i, vp]
        lib.palimpsa_step.restype = i
        lib.palimpsa_step.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, vp]
        lib.palimpsa_step_sequence_fused.restype = i
        lib.palimpsa_step_sequence_fused.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, u,
                                                     i, vp]
        lib.palimpsa_step_sequence.restype = i
        lib.palimpsa_step_sequence.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp]
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
        lib.palimpsa_set_step_l2_keep_bytes.restype = None
        lib.palimpsa_set_step_l2_keep_bytes.argtypes = [ctypes.c_longlong]
        lib.palimpsa_set_scratch_retention.restype = i
        lib.palimpsa_set_scratch_retention.argtypes = [ctypes.c_ulonglong]
        lib.palimpsa_release_scratch.restype = i
        lib.palimpsa_release_scratch.argtypes = []
        lib.palimpsa_scratch_reserved_bytes.restype = i
        lib.palimpsa_scratch_reserved_bytes.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
        lib.palimpsa_probe_issue_rate.restype = i
        lib.palimpsa_probe_issue_rate.argtypes = [i, ctypes.POINTER(ctypes.c_double), vp]
        _lib = lib
        return lib


def palimpsa_forward_plan(B, H, T, d_k, d_v, *, chunk: int = 0, bf16: bool = True):
    """The forward's launch plan on the current device (see palimpsa.h): a dict
    with segments, segment_len, launches and scratch_bytes."""
    seg, sl, ln, sb = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    rc = load_library().palimpsa_forward_plan(int(B), int(H), int(T), int(d_k), int(d_v), int(chunk),
                                              PALIMPSA_BF16 if bf16 else PALIMPSA_F32, ctypes.byref(seg),
                                              ctypes.byref(sl), ctypes.byref(ln), ctypes.byref(sb))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_plan")
    return {"segments": seg.value, "segment_len": sl.value, "launches": ln.value, "scratch_bytes": sb.value}


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


def palimpsa_set_step_l2_keep_bytes(nbytes: int) -> None:
    """Bytes of the decode state each step leaves in L2 for the next, which walks
    the state the other way (0 = stream everything in one order; see palimpsa.h)."""
    load_library().palimpsa_set_step_l2_keep_bytes(int(nbytes))


def palimpsa_set_scratch_retention(nbytes: int) -> None:
    """Bytes of freed scratch every device's pool keeps mapped between calls (see palimpsa.h)."""
    rc = load_library().palimpsa_set_scratch_retention(int(nbytes))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_set_scratch_retention")


def palimpsa_release_scratch(device=None) -> None:
    """Synchronise `device` (default: the current one) and give all of its freed
    scratch back to the driver (see palimpsa.h)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = load_library().palimpsa_release_scratch()
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_release_scratch")


def palimpsa_scratch_reserved_bytes(device=None) -> int:
    """Bytes the library's scratch pool on `device` holds mapped (0 without a pool)."""
    n = ctypes.c_size_t()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        rc = load_library().palimpsa_scratch_reserved_bytes(ctypes.byref(n))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_scratch_reserved_bytes")
    return int(n.value)


PROBE_OPS = {"rcp": 0, "ex2": 1, "ffma": 2, "rsqrt": 3, "lg2": 4}


def palimpsa_probe_issue_rate(op: str, stream=None) -> float:
    """Instructions of kind `op` ("rcp", "ex2", "ffma", "rsqrt" or "lg2") one SM of the current
    device completes per clock, measured (see palimpsa.h)."""
    r = ctypes.c_double()
    rc = load_library().palimpsa_probe_issue_rate(PROBE_OPS[op], ctypes.byref(r),
                                                  ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_probe_issue_rate")
    return float(r.value)


def _stream_handle(stream) -> int:
    """The raw handle of the stream the library launches on. A caller's stream
    other than the current one first waits for the current stream, where the
    binding (and usually the caller) made the inputs and outputs."""
    if stream is None:
        stream = torch.cuda.current_stream()
    else:
        cur = torch.cuda.current_stream(stream.device)
        if cur.cuda_stream != stream.cuda_stream:
            stream.wait_stream(cur)
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
        return _forward_from_host(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, chunk, stream)
    B, H, T, d_k, d_v, dev = _check_forward_inputs(q, k, v, beta, d_t, A, I_prior, mu0, I0, ("beta", "d_t"))
    y, mu_T, I_T = _forward_outputs(B, H, T, d_k, d_v, dev, y, mu_T, I_T)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_forward_chunked(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(I0),
            _ptr(y), _ptr(mu_T), _ptr(I_T), B, H, T, d_k, d_v, int(chunk), _in_dtype(q),
            ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_chunked")
    return y, mu_T, I_T


def _check_forward_inputs(q, k, v, beta, d_t, A, I_prior, mu0, I0, names):
    """Shapes, dtypes and placement of a forward's inputs (device tensors);
    returns (B, H, T, d_k, d_v, device)."""
    if q.device.type != "cuda":
        raise ValueError("this entry point takes device tensors")
    B, H, T, d_k = q.shape
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    _check(k, "k", q.shape, q.dtype, dev)
    _check(v, "v", (B, H, T, d_v), q.dtype, dev)
    _check(beta, names[0], (B, H, T, d_v), q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(d_t, names[1], (B, H, T), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(mu0, "mu0", (B, H, d_v, d_k), f32, dev)
    _check(I0, "I0", (B, H, d_v, d_k), f32, dev)
    return B, H, T, d_k, d_v, dev


def _forward_outputs(B, H, T, d_k, d_v, dev, y, mu_T, I_T):
    f32 = torch.float32
    if y is None:
        y = torch.empty((B, H, T, d_v), dtype=f32, device=dev)
    if mu_T is None:
        mu_T = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev)
    if I_T is None:
        I_T = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev)
    _check(y, "y", (B, H, T, d_v), f32, dev)
    _check(mu_T, "mu_T", (B, H, d_v, d_k), f32, dev)
    _check(I_T, "I_T", (B, H, d_v, d_k), f32, dev)
    return y, mu_T, I_T


def _fuse_flags(qk_norm, v_star):
    return (PALIMPSA_FUSE_QK_NORM if qk_norm else 0) | (PALIMPSA_FUSE_V_STAR if v_star else 0)


def palimpsa_forward_varlen(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0=None, I0=None, *, max_seqlen=None,
                            y=None, mu_T=None, I_T=None, chunk: int = 0, stream=None):
    """The forward over a packed batch of N sequences (see palimpsa.h).

    q, k [H, total_T, d_k] and v, beta [H, total_T, d_v] (one dtype), d_t
    [H, total_T] fp32; cu_seqlens [N + 1] int32 (sequence n = tokens
    [cu[n], cu[n+1])), on the device or the host (then copied); mu0, I0 [N, H,
    d_v, d_k] or None. max_seqlen: the longest sequence (read from cu_seqlens
    when not given, which synchronises). Device tensors otherwise. Returns
    (y [H, total_T, d_v], mu_T [N, H, d_v, d_k], I_T)."""
    return _varlen(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0, I0, max_seqlen, y, mu_T, I_T, chunk, stream,
                   None)


def palimpsa_forward_varlen_fused(q, k, v, beta_raw, d_raw, A, I_prior, cu_seqlens, b_scale=None, mu0=None, I0=None, *,
                                  qk_norm=False, v_star=False, max_seqlen=None, y=None, mu_T=None, I_T=None,
                                  chunk: int = 0, stream=None):
    """palimpsa_forward_varlen from raw projections with the fused prologue of
    palimpsa_forward_fused (see palimpsa.h)."""
    return _varlen(q, k, v, beta_raw, d_raw, A, I_prior, cu_seqlens, mu0, I0, max_seqlen, y, mu_T, I_T, chunk, stream,
                   (b_scale, _fuse_flags(qk_norm, v_star)))


def _packed_offsets(cu_seqlens, max_seqlen, dev, stream=None):
    """(offsets on the device, N, max_seqlen) of a packed batch. Host offsets are
    copied on the stream the library will use, and the copy is recorded there so
    that the allocator keeps it until that stream is done with it."""
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor of N + 1 offsets")
    N = cu_seqlens.numel() - 1
    if max_seqlen is None:
        host = cu_seqlens.cpu()
        max_seqlen = int((host[1:] - host[:-1]).max())
    if cu_seqlens.is_cuda:
        cu_d = cu_seqlens
    else:
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        with torch.cuda.stream(st):
            cu_d = cu_seqlens.to(dev, non_blocking=False)
        cu_d.record_stream(st)
    _check(cu_d, "cu_seqlens", (N + 1,), torch.int32, dev)
    return cu_d, N, int(max_seqlen)


def _varlen(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0, I0, max_seqlen, y, mu_T, I_T, chunk, stream, fused,
            ckpt=None):
    if q.device.type != "cuda":
        raise ValueError("the packed forward takes device tensors")
    H, total_T, d_k = q.shape
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    cu_d, N, max_seqlen = _packed_offsets(cu_seqlens, max_seqlen, dev, stream)
    names = ("beta", "d_t") if fused is None else ("beta_raw", "d_raw")
    _check(k, "k", q.shape, q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(v, "v", (H, total_T, d_v), q.dtype, dev)
    _check(beta, names[0], (H, total_T, d_v), q.dtype, dev)
    _check(d_t, names[1], (H, total_T), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(mu0, "mu0", (N, H, d_v, d_k), f32, dev)
    _check(I0, "I0", (N, H, d_v, d_k), f32, dev)
    y = torch.zeros((H, total_T, d_v), dtype=f32, device=dev) if y is None else y
    mu_T = torch.empty((N, H, d_v, d_k), dtype=f32, device=dev) if mu_T is None else mu_T
    I_T = torch.empty((N, H, d_v, d_k), dtype=f32, device=dev) if I_T is None else I_T
    _check(y, "y", (H, total_T, d_v), f32, dev)
    _check(mu_T, "mu_T", (N, H, d_v, d_k), f32, dev)
    _check(I_T, "I_T", (N, H, d_v, d_k), f32, dev)
    lib = load_library()
    head = [_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior)]
    mid = [_ptr(mu0), _ptr(I0), _ptr(y), _ptr(mu_T), _ptr(I_T), _ptr(cu_d), N, H, total_T, max_seqlen, d_k, d_v,
           int(chunk)]
    st = ctypes.c_void_p(_stream_handle(stream))
    with torch.cuda.device(dev):
        if ckpt is not None:
            _check(ckpt, "ckpt", packed_checkpoint_shape(N, H, total_T, d_k, d_v), f32, dev)
            mid.insert(5, _ptr(ckpt))
            rc, name = (lib.palimpsa_forward_varlen_checkpointed(*head, *mid, _in_dtype(q), st),
                        "palimpsa_forward_varlen_checkpointed")
        elif fused is None:
            rc, name = lib.palimpsa_forward_varlen(*head, *mid, _in_dtype(q), st), "palimpsa_forward_varlen"
        else:
            b_scale, flags = fused
            _check(b_scale, "b_scale", (H,), f32, dev)
            rc, name = (lib.palimpsa_forward_varlen_fused(*head, _ptr(b_scale), *mid, flags, _in_dtype(q), st),
                        "palimpsa_forward_varlen_fused")
    if rc != 0:
        raise PalimpsaError(rc, name)
    return y, mu_T, I_T


def palimpsa_segment_summary(q, k, v, beta, d_t, A, I_prior, *, summary=None, gamma=None, chunk: int = 0,
                             stream=None):
    """Summary of each head's T tokens from a zero state (see palimpsa.h):
    returns (summary [B,H,2,d_v,d_k] = (dM, dIbar), gamma [B,H] = prod alpha).
    Device tensors laid out as for palimpsa_forward_chunked."""
    B, H, T, d_k, d_v, dev = _check_forward_inputs(q, k, v, beta, d_t, A, I_prior, None, None, ("beta", "d_t"))
    f32 = torch.float32
    summary = torch.empty((B, H, 2, d_v, d_k), dtype=f32, device=dev) if summary is None else summary
    gamma = torch.empty((B, H), dtype=f32, device=dev) if gamma is None else gamma
    _check(summary, "summary", (B, H, 2, d_v, d_k), f32, dev)
    _check(gamma, "gamma", (B, H), f32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_segment_summary(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior),
                                          _ptr(summary), _ptr(gamma), B, H, T, d_k, d_v, int(chunk), _in_dtype(q),
                                          ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_segment_summary")
    return summary, gamma


def palimpsa_state_combine(summaries, gammas, I_prior, mu0=None, I0=None, *, mu_out=None, I_out=None, stream=None):
    """The state after R stretches, in order, from (mu0, I0) (see palimpsa.h):
    summaries [R,B,H,2,d_v,d_k], gammas [R,B,H] -> (mu [B,H,d_v,d_k], I)."""
    R, B, H, _, d_v, d_k = summaries.shape
    dev = summaries.device
    f32 = torch.float32
    if dev.type != "cuda":
        raise ValueError("palimpsa_state_combine takes device tensors")
    _check(summaries, "summaries", (R, B, H, 2, d_v, d_k), f32, dev)
    _check(gammas, "gammas", (R, B, H), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(mu0, "mu0", (B, H, d_v, d_k), f32, dev)
    _check(I0, "I0", (B, H, d_v, d_k), f32, dev)
    mu_out = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev) if mu_out is None else mu_out
    I_out = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev) if I_out is None else I_out
    _check(mu_out, "mu_out", (B, H, d_v, d_k), f32, dev)
    _check(I_out, "I_out", (B, H, d_v, d_k), f32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_state_combine(_ptr(summaries) if R else None, _ptr(gammas) if R else None, R,
                                        _ptr(I_prior), _ptr(mu0), _ptr(I0), _ptr(mu_out), _ptr(I_out), B, H, d_k,
                                        d_v, ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_state_combine")
    return mu_out, I_out


def palimpsa_forward_fused(q, k, v, beta_raw, d_raw, A, I_prior, b_scale=None, mu0=None, I0=None, *,
                           qk_norm=False, v_star=False, y=None, mu_T=None, I_T=None, chunk: int = 0, stream=None):
    """The forward with the layer prologue fused in (see palimpsa.h): d_t =
    softplus(d_raw), beta = b_scale * sigmoid(beta_raw), q/k L2-normalised per
    token when qk_norm, v taken as v* = beta v when v_star. Device tensors;
    b_scale [H] fp32 or None. Returns (y, mu_T, I_T)."""
    B, H, T, d_k, d_v, dev = _check_forward_inputs(q, k, v, beta_raw, d_raw, A, I_prior, mu0, I0,
                                                   ("beta_raw", "d_raw"))
    _check(b_scale, "b_scale", (H,), torch.float32, dev)
    y, mu_T, I_T = _forward_outputs(B, H, T, d_k, d_v, dev, y, mu_T, I_T)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_forward_fused(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta_raw), _ptr(d_raw), _ptr(A), _ptr(I_prior), _ptr(b_scale), _ptr(mu0),
            _ptr(I0), _ptr(y), _ptr(mu_T), _ptr(I_T), B, H, T, d_k, d_v, int(chunk), _fuse_flags(qk_norm, v_star),
            _in_dtype(q), ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_fused")
    return y, mu_T, I_T


def palimpsa_step_fused(q, k, v, beta_raw, d_raw, A, I_prior, mu, I, b_scale=None, *, qk_norm=False, v_star=False,
                        y=None, stream=None):
    """Decode tokens from raw inputs (see palimpsa.h); mu, I updated in place.
    Device tensors. One token: q, k [B,H,d_k], v and beta_raw [B,H,d_v], d_raw
    [B,H] -> y [B,H,d_v]. S tokens: a leading steps dimension on q, k, v,
    beta_raw, d_raw -> y [S,B,H,d_v], enqueued by one palimpsa_step_sequence_fused
    call."""
    if q.device.type != "cuda":
        raise ValueError("palimpsa_step_fused takes device tensors")
    seq = q.dim() == 4
    lead = (q.shape[0],) if seq else ()
    B, H, d_k = q.shape[-3:]
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    _check(k, "k", q.shape, q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(v, "v", lead + (B, H, d_v), q.dtype, dev)
    _check(beta_raw, "beta_raw", lead + (B, H, d_v), q.dtype, dev)
    _check(d_raw, "d_raw", lead + (B, H), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    _check(b_scale, "b_scale", (H,), f32, dev)
    _check(mu, "mu", (B, H, d_v, d_k), f32, dev)
    _check(I, "I", (B, H, d_v, d_k), f32, dev)
    y = torch.empty(lead + (B, H, d_v), dtype=f32, device=dev) if y is None else y
    _check(y, "y", lead + (B, H, d_v), f32, dev)
    lib = load_library()
    head = [_ptr(q), _ptr(k), _ptr(v), _ptr(beta_raw), _ptr(d_raw), _ptr(A), _ptr(I_prior), _ptr(b_scale), _ptr(mu),
            _ptr(I), _ptr(y)]
    tail = [B, H, d_k, d_v, _fuse_flags(qk_norm, v_star), _in_dtype(q), ctypes.c_void_p(_stream_handle(stream))]
    with torch.cuda.device(dev):
        if seq:
            rc, name = lib.palimpsa_step_sequence_fused(*head, int(q.shape[0]), *tail), "palimpsa_step_sequence_fused"
        else:
            rc, name = lib.palimpsa_step_fused(*head, *tail), "palimpsa_step_fused"
    if rc != 0:
        raise PalimpsaError(rc, name)
    return y


def palimpsa_forward_without_meta(q, k, v, beta, d_t, A, I_prior, mu0=None, *, y=None, mu_T=None, chunk: int = 0,
                                  stream=None):
    """The "without Meta" comparator (see palimpsa.h): importance frozen at I_prior.
    Device tensors only. Returns (y, mu_T)."""
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
    y = torch.empty((B, H, T, d_v), dtype=f32, device=dev) if y is None else y
    mu_T = torch.empty((B, H, d_v, d_k), dtype=f32, device=dev) if mu_T is None else mu_T
    _check(y, "y", (B, H, T, d_v), f32, dev)
    _check(mu_T, "mu_T", (B, H, d_v, d_k), f32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_forward_without_meta(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(y),
            _ptr(mu_T), B, H, T, d_k, d_v, int(chunk), _in_dtype(q), ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_without_meta")
    return y, mu_T


def palimpsa_checkpoint_bytes(B, H, T, d_k, d_v) -> int:
    """Bytes of the training checkpoints of a forward of these sizes (see palimpsa.h)."""
    return int(load_library().palimpsa_checkpoint_bytes(int(B), int(H), int(T), int(d_k), int(d_v)))


def palimpsa_forward_checkpointed(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None, *, ckpt=None, y=None,
                                  mu_T=None, I_T=None, chunk: int = 0, stream=None):
    """The forward for training (see palimpsa.h): palimpsa_forward_chunked that also
    writes the state before every 32nd token, for palimpsa_backward(ckpt=...).
    Device tensors. Returns (y, mu_T, I_T, ckpt); ckpt is [B,H,ceil(T/32),d_v,2,d_k]."""
    B, H, T, d_k, d_v, dev = _check_forward_inputs(q, k, v, beta, d_t, A, I_prior, mu0, I0, ("beta", "d_t"))
    y, mu_T, I_T = _forward_outputs(B, H, T, d_k, d_v, dev, y, mu_T, I_T)
    shape = (B, H, -(-T // 32), d_v, 2, d_k)
    ckpt = torch.empty(shape, dtype=torch.float32, device=dev) if ckpt is None else ckpt
    _check(ckpt, "ckpt", shape, torch.float32, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_forward_checkpointed(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(I0), _ptr(y),
            _ptr(mu_T), _ptr(I_T), _ptr(ckpt), B, H, T, d_k, d_v, int(chunk), _in_dtype(q),
            ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_forward_checkpointed")
    return y, mu_T, I_T, ckpt


def palimpsa_backward(q, k, v, beta, d_t, A, I_prior, mu0, I0, dy, dmu_T=None, dI_T=None, *, want_state_grads=True,
                      ckpt=None, stream=None):
    """Gradients through palimpsa_forward_chunked (see palimpsa.h). Device tensors.
    With ckpt (from palimpsa_forward_checkpointed on the same inputs) the
    backward reads the states instead of recomputing them.

    Returns a dict: dq, dk, dv, dbeta, dd_t, dA, dI_prior, and dmu0 / dI0 when
    want_state_grads (fp32 throughout)."""
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
    for name, t in (("mu0", mu0), ("I0", I0), ("dmu_T", dmu_T), ("dI_T", dI_T)):
        _check(t, name, (B, H, d_v, d_k), f32, dev)
    _check(dy, "dy", (B, H, T, d_v), f32, dev)
    e = lambda *shape: torch.empty(shape, dtype=f32, device=dev)
    g = {"dq": e(B, H, T, d_k), "dk": e(B, H, T, d_k), "dv": e(B, H, T, d_v), "dbeta": e(B, H, T, d_v),
         "dd_t": e(B, H, T), "dA": e(H), "dI_prior": e(H)}
    if want_state_grads:
        g["dmu0"] = e(B, H, d_v, d_k)
        g["dI0"] = e(B, H, d_v, d_k)
    lib = load_library()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(I0), _ptr(dy),
            _ptr(dmu_T), _ptr(dI_T), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dbeta"]), _ptr(g["dd_t"]),
            _ptr(g["dA"]), _ptr(g["dI_prior"]), _ptr(g.get("dmu0")), _ptr(g.get("dI0"))]
    tail = [B, H, T, d_k, d_v, _in_dtype(q), ctypes.c_void_p(_stream_handle(stream))]
    with torch.cuda.device(dev):
        if ckpt is None:
            rc, name = lib.palimpsa_backward(*args, *tail), "palimpsa_backward"
        else:
            _check(ckpt, "ckpt", (B, H, -(-T // 32), d_v, 2, d_k), f32, dev)
            rc, name = lib.palimpsa_backward_checkpointed(*args, _ptr(ckpt), *tail), "palimpsa_backward_checkpointed"
    if rc != 0:
        raise PalimpsaError(rc, name)
    return g


def palimpsa_checkpoint_bytes_varlen(N, H, total_T, d_k, d_v) -> int:
    """Bytes of the training checkpoints of a packed forward (see palimpsa.h)."""
    return int(load_library().palimpsa_checkpoint_bytes_varlen(int(N), int(H), int(total_T), int(d_k), int(d_v)))


def packed_checkpoint_shape(N, H, total_T, d_k, d_v):
    """Shape of a packed batch's checkpoints: per head, total_T // 32 + N slots."""
    return (H, total_T // 32 + N, d_v, 2, d_k)


def palimpsa_forward_varlen_checkpointed(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0=None, I0=None, *,
                                         max_seqlen=None, ckpt=None, y=None, mu_T=None, I_T=None, chunk: int = 0,
                                         stream=None):
    """palimpsa_forward_varlen for training (see palimpsa.h): also writes each
    sequence's state before its every 32nd token, for palimpsa_backward_varlen.
    Returns (y, mu_T, I_T, ckpt); ckpt is [H, total_T//32 + N, d_v, 2, d_k], and
    sequence n (from token s0) keeps its checkpoint c in slot s0//32 + n + c."""
    if q.device.type != "cuda":
        raise ValueError("the packed forward takes device tensors")
    cu_d, N, max_seqlen = _packed_offsets(cu_seqlens, max_seqlen, q.device, stream)
    H, total_T, d_k = q.shape
    d_v = v.shape[-1]
    if ckpt is None:
        ckpt = torch.empty(packed_checkpoint_shape(N, H, total_T, d_k, d_v), dtype=torch.float32, device=q.device)
    y, mu_T, I_T = _varlen(q, k, v, beta, d_t, A, I_prior, cu_d, mu0, I0, max_seqlen, y, mu_T, I_T, chunk, stream,
                           None, ckpt=ckpt)
    return y, mu_T, I_T, ckpt


def palimpsa_backward_varlen(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0, I0, dy, dmu_T=None, dI_T=None, *,
                             max_seqlen=None, want_state_grads=True, ckpt=None, stream=None):
    """Gradients through palimpsa_forward_varlen (see palimpsa.h). Device
    tensors in the packed layout; ckpt from palimpsa_forward_varlen_checkpointed
    on the same inputs, or None to recompute the states.

    Returns a dict as palimpsa_backward: dq, dk [H,total_T,d_k], dv, dbeta
    [H,total_T,d_v], dd_t [H,total_T], dA, dI_prior [H] (summed over the
    sequences), and dmu0 / dI0 [N,H,d_v,d_k] when want_state_grads. Rows of
    tokens outside every sequence are zero."""
    if q.device.type != "cuda":
        raise ValueError("the packed backward takes device tensors")
    H, total_T, d_k = q.shape
    d_v = v.shape[-1]
    dev = q.device
    f32 = torch.float32
    cu_d, N, max_seqlen = _packed_offsets(cu_seqlens, max_seqlen, dev, stream)
    _check(k, "k", q.shape, q.dtype, dev)
    _check(q, "q", q.shape, None, dev)
    _check(v, "v", (H, total_T, d_v), q.dtype, dev)
    _check(beta, "beta", (H, total_T, d_v), q.dtype, dev)
    _check(d_t, "d_t", (H, total_T), f32, dev)
    _check(A, "A", (H,), f32, dev)
    _check(I_prior, "I_prior", (H,), f32, dev)
    for name, t in (("mu0", mu0), ("I0", I0), ("dmu_T", dmu_T), ("dI_T", dI_T)):
        _check(t, name, (N, H, d_v, d_k), f32, dev)
    _check(dy, "dy", (H, total_T, d_v), f32, dev)
    _check(ckpt, "ckpt", packed_checkpoint_shape(N, H, total_T, d_k, d_v), f32, dev)
    e = lambda *shape: torch.empty(shape, dtype=f32, device=dev)
    z = lambda *shape: torch.zeros(shape, dtype=f32, device=dev)
    # dq, dk, dd_t are zeroed by the library; dv, dbeta only where a sequence is
    g = {"dq": e(H, total_T, d_k), "dk": e(H, total_T, d_k), "dv": z(H, total_T, d_v), "dbeta": z(H, total_T, d_v),
         "dd_t": e(H, total_T), "dA": e(H), "dI_prior": e(H)}
    if want_state_grads:
        g["dmu0"] = e(N, H, d_v, d_k)
        g["dI0"] = e(N, H, d_v, d_k)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.palimpsa_backward_varlen(
            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu0), _ptr(I0), _ptr(dy),
            _ptr(dmu_T), _ptr(dI_T), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dbeta"]), _ptr(g["dd_t"]),
            _ptr(g["dA"]), _ptr(g["dI_prior"]), _ptr(g.get("dmu0")), _ptr(g.get("dI0")), _ptr(ckpt), _ptr(cu_d),
            N, H, total_T, max_seqlen, d_k, d_v, _in_dtype(q), ctypes.c_void_p(_stream_handle(stream)))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_backward_varlen")
    return g


def palimpsa_step(q, k, v, beta, d_t, A, I_prior, mu, I, *, y=None, stream=None):
    """Decode tokens (see palimpsa.h): updates mu, I in place and returns y.

    One token: q, k [B,H,d_k], v, beta [B,H,d_v], d_t [B,H] -> y [B,H,d_v].
    A sequence of S tokens: a leading steps dimension on q, k, v, beta, d_t
    -> y [S,B,H,d_v]; the tokens go in order, enqueued by one palimpsa_step_sequence
    call (device inputs) or by blocks of tokens streamed from the host (host inputs)."""
    if q.dim() == 4:
        return _step_sequence(q, k, v, beta, d_t, A, I_prior, mu, I, y, stream)
    if q.device.type == "cpu":
        # Host inputs: the state stays where it is when it is on the device (the
        # resident decode state); host state is copied in and back.
        # Every copy and the step run on one stream, in order.
        dev = _compute_device(mu, I, y)
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        with torch.cuda.device(dev), torch.cuda.stream(st):
            dq = _to_device([q, k, v, beta, d_t, A, I_prior, mu, I], dev)
            ydev = y if (y is not None and y.is_cuda) else None
            ry = palimpsa_step(*dq, y=ydev, stream=st)
            if not mu.is_cuda:
                mu.copy_(dq[7], non_blocking=True)
            if not I.is_cuda:
                I.copy_(dq[8], non_blocking=True)
            out = _deliver(y, ry)
        st.synchronize()
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


# ---------------------------------------------------------------- host-buffer pipelines
#
# Callers with host (ideally pinned) buffers: the work is cut into blocks that
# move through three CUDA streams - host-to-device copies, the library's
# kernels on the caller's stream, device-to-host copies - two device buffers
# deep, so the copies of one block overlap the computation of its neighbours.
# Only copies and stream/event ordering happen here; all arithmetic runs in
# the library's kernels. The call returns when every result is in place.

HOST_BLOCK_BYTES = 256 << 20   # host input bytes per pipelined block


# Each pipelined forward launch covers at least this many heads, about eight
# waves of CTAs on a 152-SM part: a launch of few waves pays a partial last wave.
MIN_HEADS_PER_FORWARD_BLOCK = 2432


def _blocks(n, per_item_bytes, target=None, min_items=1):
    target = HOST_BLOCK_BYTES if target is None else target
    size = max(1, min_items, min(n, target // max(1, per_item_bytes)))
    size = min(size, max(1, n))
    return [(i, min(n, i + size)) for i in range(0, n, size)], size


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


class _Pipe:
    def __init__(self, dev, stream):
        self.dev = dev
        self.comp = stream or torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.in_free = [None, None]    # compute finished reading slot s
        self.out_free = [None, None]   # device-to-host copy finished reading slot s

    def load(self, slot, pairs):
        """Copy (device_dst, host_src) pairs on the h2d stream into slot `slot`."""
        if self.in_free[slot] is not None:
            self.h2d.wait_event(self.in_free[slot])
        with torch.cuda.stream(self.h2d):
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(self.h2d)
        self.comp.wait_event(ev)
        if self.out_free[slot] is not None:
            self.comp.wait_event(self.out_free[slot])

    def computed(self, slot):
        ev = torch.cuda.Event()
        ev.record(self.comp)
        self.in_free[slot] = ev
        return ev

    def store(self, slot, after, pairs):
        """Copy (host_dst, device_src) pairs on the d2h stream once `after` has fired."""
        self.d2h.wait_event(after)
        with torch.cuda.stream(self.d2h):
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(self.d2h)
        self.out_free[slot] = ev

    def finish(self):
        self.d2h.synchronize()
        self.h2d.synchronize()
        self.comp.synchronize()


def _host_out(t, shape, dtype):
    return t if t is not None else torch.empty(shape, dtype=dtype, pin_memory=True)


def _forward_from_host(q, k, v, beta, d_t, A, I_prior, mu0, I0, y, mu_T, I_T, chunk, stream):
    """palimpsa_forward_chunked with host inputs: pipelined over batch blocks
    (heads of different batch entries are independent)."""
    dev = _compute_device(y, mu_T, I_T, mu0, I0)
    B, H, T, d_k = q.shape
    d_v = v.shape[-1]
    f32 = torch.float32
    per_b = sum(_nbytes(t) // max(1, B) for t in (q, k, v, beta, d_t, mu0, I0))
    blocks, nb = _blocks(B, per_b, min_items=-(-MIN_HEADS_PER_FORWARD_BLOCK // max(1, H)))
    outs = []
    for t, shape in ((y, (B, H, T, d_v)), (mu_T, (B, H, d_v, d_k)), (I_T, (B, H, d_v, d_k))):
        outs.append(t if (t is not None and t.is_cuda) else _host_out(t, shape, f32))
    with torch.cuda.device(dev):
        p = _Pipe(dev, stream)
        with torch.cuda.stream(p.comp):
            A_d = A.to(dev, non_blocking=True) if not A.is_cuda else A
            Ip_d = I_prior.to(dev, non_blocking=True) if not I_prior.is_cuda else I_prior
        ins = [q, k, v, beta, d_t, mu0, I0]
        slots = [[None if t is None else torch.empty((nb,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
                  for t in ins] for _ in range(min(2, len(blocks)))]
        oslots = [[None if o.is_cuda else torch.empty((nb,) + tuple(o.shape[1:]), dtype=f32, device=dev)
                   for o in outs] for _ in range(min(2, len(blocks)))]
        for i, (b0, b1) in enumerate(blocks):
            s, n = i % 2, b1 - b0
            src = [None if t is None else (t[b0:b1] if t.is_cuda else None) for t in ins]
            pairs = []
            dq = []
            for j, t in enumerate(ins):
                if t is None:
                    dq.append(None)
                elif t.is_cuda:
                    dq.append(src[j])
                else:
                    dq.append(slots[s][j][:n])
                    pairs.append((dq[-1], t[b0:b1]))
            p.load(s, pairs)
            od = [o[b0:b1] if o.is_cuda else oslots[s][j][:n] for j, o in enumerate(outs)]
            palimpsa_forward_chunked(dq[0], dq[1], dq[2], dq[3], dq[4], A_d, Ip_d, dq[5], dq[6], y=od[0],
                                     mu_T=od[1], I_T=od[2], chunk=chunk, stream=p.comp)
            ev = p.computed(s)
            p.store(s, ev, [(o[b0:b1], od[j]) for j, o in enumerate(outs) if not o.is_cuda])
        p.finish()
    return tuple(outs)


def _steps_direct(q, k, v, beta, d_t, A, I_prior, mu, I, y, n, stream_handle):
    """The first n tokens of contiguous device tensors whose leading index is the
    token (validated by the caller), as one palimpsa_step_sequence call: the
    library enqueues the n step launches itself."""
    _, B, H, d_k = q.shape
    d_v = v.shape[-1]
    rc = load_library().palimpsa_step_sequence(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(I_prior), _ptr(mu), _ptr(I), _ptr(y), int(n),
        B, H, d_k, d_v, _in_dtype(q), ctypes.c_void_p(stream_handle))
    if rc != 0:
        raise PalimpsaError(rc, "palimpsa_step_sequence")


def _step_sequence(q, k, v, beta, d_t, A, I_prior, mu, I, y, stream):
    """S decode tokens in order; host inputs are pipelined over blocks of tokens
    while the state stays resident on the device."""
    S, B, H, d_k = q.shape
    d_v = v.shape[-1]
    f32 = torch.float32
    if q.device.type != "cpu":
        dev = q.device
        _check(k, "k", q.shape, q.dtype, dev)
        _check(q, "q", q.shape, None, dev)
        _check(v, "v", (S, B, H, d_v), q.dtype, dev)
        _check(beta, "beta", (S, B, H, d_v), q.dtype, dev)
        _check(d_t, "d_t", (S, B, H), f32, dev)
        _check(A, "A", (H,), f32, dev)
        _check(I_prior, "I_prior", (H,), f32, dev)
        _check(mu, "mu", (B, H, d_v, d_k), f32, dev)
        _check(I, "I", (B, H, d_v, d_k), f32, dev)
        y = torch.empty((S, B, H, d_v), dtype=f32, device=dev) if y is None else y
        _check(y, "y", (S, B, H, d_v), f32, dev)
        with torch.cuda.device(dev):
            _steps_direct(q, k, v, beta, d_t, A, I_prior, mu, I, y, S, _stream_handle(stream))
        return y
    dev = _compute_device(mu, I, y)
    _check(k, "k", q.shape, q.dtype)
    _check(q, "q", q.shape)
    _check(v, "v", (S, B, H, d_v), q.dtype)
    _check(beta, "beta", (S, B, H, d_v), q.dtype)
    _check(d_t, "d_t", (S, B, H), f32)
    _check(A, "A", (H,), f32)
    _check(I_prior, "I_prior", (H,), f32)
    _check(mu, "mu", (B, H, d_v, d_k), f32)
    _check(I, "I", (B, H, d_v, d_k), f32)
    _check(y, "y", (S, B, H, d_v), f32)
    _in_dtype(q)
    per_step = sum(_nbytes(t) // max(1, S) for t in (q, k, v, beta, d_t))
    blocks, ns = _blocks(S, per_step)
    y_dev_direct = y is not None and y.is_cuda
    y = y if y is not None else torch.empty((S, B, H, d_v), dtype=f32, pin_memory=True)
    with torch.cuda.device(dev):
        p = _Pipe(dev, stream)
        with torch.cuda.stream(p.comp):
            A_d = A.to(dev, non_blocking=True) if not A.is_cuda else A
            Ip_d = I_prior.to(dev, non_blocking=True) if not I_prior.is_cuda else I_prior
            mu_d = mu if mu.is_cuda else mu.to(dev, non_blocking=True)
            I_d = I if I.is_cuda else I.to(dev, non_blocking=True)
        ins = [q, k, v, beta, d_t]
        slots = [[torch.empty((ns,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev) for t in ins]
                 for _ in range(min(2, len(blocks)))]
        yslots = [torch.empty((ns, B, H, d_v), dtype=f32, device=dev) for _ in range(min(2, len(blocks)))]
        for i, (s0, s1) in enumerate(blocks):
            s, n = i % 2, s1 - s0
            p.load(s, [(slots[s][j][:n], t[s0:s1]) for j, t in enumerate(ins)])
            yd = y[s0:s1] if y_dev_direct else yslots[s][:n]
            _steps_direct(*slots[s], A_d, Ip_d, mu_d, I_d, yd, n, p.comp.cuda_stream)
            ev = p.computed(s)
            if not y_dev_direct:
                p.store(s, ev, [(y[s0:s1], yd)])
        if not mu.is_cuda:
            with torch.cuda.stream(p.comp):
                mu.copy_(mu_d, non_blocking=True)
                I.copy_(I_d, non_blocking=True)
        p.finish()
    return y
