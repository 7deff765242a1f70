"""ORACLE — test infrastructure only (see ``oracle/__init__``).

Variable-length batches in fp64: N independent sequences of different lengths,
packed one after another along the token axis, each with its own initial and
final state. Only ``tests/``, the smoke check and the benchmark's CPU-baseline
leg may use it.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — the recurrence runs per sequence from that
sequence's initial state (slide 7 / Eq. (5), slide 9: the state is carried
from chunk to chunk within a sequence). A packed batch is by definition the
same as running every sequence on its own, which is what this does: one
``oracle.forward`` call per sequence on its slice of the packed tensors.

Packed layout (the dense layout with B = 1 and the sequences concatenated
along T): q, k [H, total_T, dk]; v, beta [H, total_T, dv]; d_t [H, total_T];
cu_seqlens [N + 1] non-decreasing, sequence n = tokens [cu[n], cu[n+1]);
mu0, I0, mu_T, I_T [N, H, dv, dk]. Tokens outside every sequence are not read
and their y rows are left at zero.
"""
from __future__ import annotations

import numpy as np

import oracle


def forward(q, k, v, beta, d_t, A, I_prior, cu_seqlens, mu0=None, I0=None, nthreads: int = 0, v_star=False):
    """Returns (y [H, total_T, dv], mu_T [N, H, dv, dk], I_T [N, H, dv, dk]) in fp64."""
    q, k, v, beta, d_t = (np.asarray(x, dtype=np.float64) for x in (q, k, v, beta, d_t))
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    H, total_T, dk = q.shape
    dv = v.shape[-1]
    y = np.zeros((H, total_T, dv))
    muT = np.zeros((N, H, dv, dk))
    IT = np.zeros((N, H, dv, dk))
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        m0 = None if mu0 is None else np.asarray(mu0, dtype=np.float64)[n:n + 1]
        i0 = None if I0 is None else np.asarray(I0, dtype=np.float64)[n:n + 1]
        yn, mn, In = oracle.forward(q[None, :, s0:s1], k[None, :, s0:s1], v[None, :, s0:s1], beta[None, :, s0:s1],
                                    d_t[None, :, s0:s1], A, I_prior, mu0=m0, I0=i0, nthreads=nthreads,
                                    v_star=v_star)
        y[:, s0:s1] = yn[0]
        muT[n], IT[n] = mn[0], In[0]
    return y, muT, IT
