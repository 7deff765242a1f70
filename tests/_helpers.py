"""Shared test helpers: relative-L2 error, oracle runs on torch inputs, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from metaplastic_linear_attention_gb300.synthetic import as_float64_numpy

# Relative-L2 bars (the target tolerances): fp32 inputs 1e-4; bf16 inputs with
# fp32 state 2e-2 (the oracle consumes the same bf16-rounded values, so the GPU
# is in practice far inside the bf16 bar; TIGHT records that stronger claim).
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
TIGHT = 1e-4


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def tol_for(inputs) -> float:
    return TOL_BF16 if inputs["q"].dtype == torch.bfloat16 else TOL_F32


def oracle_forward_from(inputs, mu0=None, I0=None, heads=None, nthreads=0):
    """Run the fp64 oracle on (a subset of heads of) torch inputs.

    heads: optional list of (b, h) pairs; the result then has B = 1, H = len(heads)
    (A and I_prior are gathered per pair)."""
    f = as_float64_numpy
    q, k, v, beta, d_t = (f(inputs[n]) for n in ("q", "k", "v", "beta", "d_t"))
    A, Ip = f(inputs["A"]), f(inputs["I_prior"])
    m0 = None if mu0 is None else f(mu0)
    i0 = None if I0 is None else f(I0)
    if heads is not None:
        bs = [b for b, _ in heads]
        hs = [h for _, h in heads]
        q, k, v, beta, d_t = (x[bs, hs][None] for x in (q, k, v, beta, d_t))
        A, Ip = A[hs], Ip[hs]
        m0 = None if m0 is None else m0[bs, hs][None]
        i0 = None if i0 is None else i0[bs, hs][None]
    return oracle.forward(q, k, v, beta, d_t, A, Ip, mu0=m0, I0=i0, nthreads=nthreads)


def pick(t: torch.Tensor, heads):
    """Gather [B, H, ...] tensor rows for (b, h) pairs -> numpy [1, n, ...]."""
    bs = [b for b, _ in heads]
    hs = [h for _, h in heads]
    return as_float64_numpy(t)[bs, hs][None]
