"""ORACLE — test infrastructure only (see ``oracle/__init__``).

The fused layer prologue in fp64: what turns a layer's raw projections into
the recurrence's inputs before Eq. (5) runs. Only ``tests/``, the smoke check
and the benchmark's CPU-baseline leg may use it.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models":
* slide 10 (paper Sec. 2.2, App. A.1): the Palimpsa-D block L2-normalises
  queries and keys (Palimpsa-M does not);
* slide 11 (Secs. 2.3-2.4) and reading notes 2.8: the kernel may take
  v* = beta (.) v itself as its input, so a small beta does not make the
  content write vanish; a per-head b_scale, fixed within a context, scales the
  importance gate;
* slide 5 and slide 4: alpha_t = exp(-A d_t) with d_t >= 0, and beta >= 0.

The pages do not print the activations that keep d_t and beta in their
domains. This statement takes the ones the workload recipes use:
d_t = softplus(d_raw) and beta = b_scale[h] * sigmoid(beta_raw). The L2 norm
divides by max(||x||_2, 1e-12), so an all-zero vector stays zero.

Each step is written out in the order above; the recurrence itself is the C
oracle (``oracle.forward`` / ``oracle.step`` with ``v_star``).
"""
from __future__ import annotations

import numpy as np

import oracle

NORM_EPS = 1e-12


def softplus(x):
    """log(1 + e^x), written as max(x, 0) + log1p(e^-|x|) so it neither
    overflows for large x nor loses the tail for very negative x."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    """1 / (1 + e^-x); e^-x may overflow to inf for x < -709, giving 0."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def l2_normalize(x):
    """x / max(||x||_2, 1e-12) over the last axis (one token's d_k values)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, NORM_EPS)


def apply(q, k, v, beta_raw, d_raw, b_scale=None, qk_norm=False):
    """Raw inputs -> the recurrence's inputs (q, k, v, beta, d_t), all fp64.

    Sequence layout: q, k [B,H,T,dk]; v, beta_raw [B,H,T,dv]; d_raw [B,H,T].
    One token: the same without T. b_scale [H] or None (meaning 1); heads are
    axis 1 in both layouts."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    beta_raw = np.asarray(beta_raw, dtype=np.float64)
    d_raw = np.asarray(d_raw, dtype=np.float64)
    if qk_norm:
        q, k = l2_normalize(q), l2_normalize(k)
    d_t = softplus(d_raw)
    beta = sigmoid(beta_raw)
    if b_scale is not None:
        bs = np.asarray(b_scale, dtype=np.float64)
        beta = beta * bs.reshape((1, bs.shape[0]) + (1,) * (beta.ndim - 2))
    return q, k, v, beta, d_t


def forward(q, k, v, beta_raw, d_raw, A, I_prior, b_scale=None, mu0=None, I0=None, qk_norm=False, v_star=False,
            nthreads: int = 0):
    """The fused forward: the prologue on [B,H,T,.] raw inputs, then Eq. (5)
    over the sequence (the M-write takes v as v* when v_star).
    Returns (y, mu_T, I_T) in fp64."""
    q, k, v, beta, d_t = apply(q, k, v, beta_raw, d_raw, b_scale, qk_norm)
    return oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0, nthreads=nthreads, v_star=v_star)


def step(q, k, v, beta_raw, d_raw, A, I_prior, mu, I, b_scale=None, qk_norm=False, v_star=False,
         nthreads: int = 0):
    """The fused decode step on one token's raw inputs: q, k [B,H,dk];
    v, beta_raw [B,H,dv]; d_raw [B,H]. Returns (y, mu', I')."""
    q, k, v, beta, d_t = apply(q, k, v, beta_raw, d_raw, b_scale, qk_norm)
    return oracle.step(q, k, v, beta, d_t, A, I_prior, mu, I, nthreads=nthreads, v_star=v_star)
