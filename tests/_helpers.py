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



U32 = 2.0 ** -24  # fp32 unit roundoff


def dA_within_bar(got_dA, ref_dA, got_dd_t, ref_dd_t, d_t, A, rel=TIGHT):
    """Per-head check of dA against the oracle, through dd_t.

    A and d_t enter the recurrence only through alpha = exp(-A d_t), so
    dA_h = sum over the head's tokens of dd_t * d_t / A_h, both for the exact
    gradients and (up to fp32 rounding) for the kernel's, which forms dd_t and dA
    from the same per-token alpha adjoint. An error in dA is then bounded by the
    error in dd_t carried through that linear map, ||delta dd_t,h|| ||d_t,h|| / A_h
    (Cauchy-Schwarz), plus the probabilistic fp32 summation bound
    4 sqrt(n) u sum|dd_t d_t| / A_h (Higham and Mary, "A new approach to
    probabilistic rounding error analysis", 2019), plus the relative bar (which
    also covers the rounding of the kernel's per-CTA partials of the map). dd_t
    itself is held to the relative bar elsewhere, so this passes dA exactly when it
    is the consistent image of a dd_t that passed, and a wrong dA term (a wrong
    token's d_t, a dropped factor) fails it. A relative bar on dA alone cannot be
    met in any precision where the exact dA vanishes by cancellation: on the first
    token from the prior state neither I nor mu depends on alpha.

    dA arrays [H]; dd_t, d_t [B, H, T] (head on axis 1) or [H, T] (axis 0); A [H].
    Returns (ok, detail)."""
    f = lambda x: np.asarray(x, dtype=np.float64)
    got, ref, gdd, rdd, dt, A = f(got_dA), f(ref_dA), f(got_dd_t), f(ref_dd_t), f(d_t), f(A)
    if dt.ndim == 3:
        gdd, rdd, dt = (np.moveaxis(x, 1, 0).reshape(x.shape[1], -1) for x in (gdd, rdd, dt))
    n = dt.shape[1]
    cs = np.linalg.norm(gdd - rdd, axis=1) * np.linalg.norm(dt, axis=1) / A
    slack = 4.0 * np.sqrt(max(n, 1)) * U32 * np.abs(gdd * dt).sum(axis=1) / A
    bar = rel * np.abs(ref) + (1.0 + rel) * cs + slack
    err = np.abs(got - ref)
    return bool(np.all(err <= bar)), dict(err=err.tolist(), bar=bar.tolist())
