"""ORACLE — test infrastructure only.

A plain, slow fp64 CPU statement of the Palimpsa dual-state recurrence
(Bonnet et al., "Learning to Remember, Learn, and Forget in Attention-Based
Models", Eq. (5) and the readout y_t = mu_t q_t). It exists to check the CUDA
library, never to stand in for it: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. It shares no code with
the CUDA path.

Contents:
* ``palimpsa_oracle.c`` — the sequential token-by-token recurrence in fp64
  (OpenMP over independent value rows only), loaded here through ctypes.
* ``prologue`` — the fused layer prologue in fp64: per-token L2 norm of q and
  k, d_t = softplus(raw), beta = b_scale * sigmoid(raw), and the v* input.
* ``varlen`` — packed variable-length batches: one ``forward`` per sequence.
* ``reference_np`` — independent NumPy statements: the mean/precision form, the
  chunked natural-parameter form and the full-Gaussian posterior it
  approximates.

Pins (what the oracle is checked against, in ``tests/test_oracle_*.py``): the
slide deck's worked examples (slide 8 scalar table, slide 25 full vs diagonal),
the discount and stationary-precision closed forms, the Mamba2 limit against a
separately written scalar-decay linear-attention sum, the coupled posterior on
axis-aligned keys, the Eq. (3) stationarity system, positivity, chunked ==
sequential, row independence, linearity in v and the prior-scale invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "palimpsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpalimpsa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, dp, dp,
                                       dp, dp, dp, L, L, L, L, L, ctypes.c_int]
        lib.oracle_forward_ex.restype = ctypes.c_int
        lib.oracle_forward_ex.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int, dp, dp,
                                          dp, dp, dp, L, L, L, L, L, ctypes.c_int]
        lib.oracle_step_ex.restype = ctypes.c_int
        lib.oracle_step_ex.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int, dp, dp, dp,
                                       L, L, L, L, ctypes.c_int]
        lib.oracle_step.restype = ctypes.c_int
        lib.oracle_step.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.c_int, dp, dp, dp,
                                    L, L, L, L, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def forward(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None, nthreads: int = 0, v_star: bool = False):
    """Sequential Eq. (5) over T tokens for every (b, h, value row).

    q, k [B,H,T,dk]; v, beta [B,H,T,dv]; d_t [B,H,T]; A [H]; I_prior [H] or
    [H,dv,dk]; mu0, I0 [B,H,dv,dk] or None (mu0 = 0, I0 = I_prior).
    With v_star, v holds v* = beta (.) v and is written as is (slide 11).
    Returns (y [B,H,T,dv], mu_T, I_T) in fp64.
    """
    q, k, v, beta, d_t, A, Ip = (_f64(x) for x in (q, k, v, beta, d_t, A, I_prior))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, H, T, dv) and beta.shape == v.shape
    assert d_t.shape == (B, H, T) and A.shape == (H,)
    prior_full = 0 if Ip.shape == (H,) else 1
    if prior_full:
        assert Ip.size == H * dv * dk
    m0 = None if mu0 is None else _f64(mu0)
    i0 = None if I0 is None else _f64(I0)
    y = np.zeros((B, H, T, dv))
    muT = np.zeros((B, H, dv, dk))
    IT = np.zeros((B, H, dv, dk))
    rc = _load().oracle_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(Ip),
                                   prior_full, int(bool(v_star)), _ptr(m0), _ptr(i0), _ptr(y), _ptr(muT),
                                   _ptr(IT), B, H, T, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_forward failed with code {rc}")
    return y, muT, IT


def step(q, k, v, beta, d_t, A, I_prior, mu, I, nthreads: int = 0, v_star: bool = False):
    """One recurrent token: q, k [B,H,dk]; v, beta [B,H,dv]; d_t [B,H]
    (v holds v* when v_star, as in ``forward``).

    Returns (y [B,H,dv], mu', I') without modifying the arguments.
    """
    q, k, v, beta, d_t, A, Ip = (_f64(x) for x in (q, k, v, beta, d_t, A, I_prior))
    B, H, dk = q.shape
    dv = v.shape[-1]
    prior_full = 0 if Ip.shape == (H,) else 1
    mu_o = _f64(mu).copy()
    I_o = _f64(I).copy()
    y = np.zeros((B, H, dv))
    rc = _load().oracle_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d_t), _ptr(A), _ptr(Ip),
                                prior_full, int(bool(v_star)), _ptr(mu_o), _ptr(I_o), _ptr(y), B, H, dk, dv,
                                int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_step failed with code {rc}")
    return y, mu_o, I_o
