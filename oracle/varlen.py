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

Gradients (``gradients``) follow from the same definition: the packed loss is
the sum of the per-sequence losses, so each sequence's input gradients are
those of the recurrence run on it alone (``oracle.autograd``), and the shared
per-head parameters A and I_prior collect the sum over sequences.

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


def gradients(inputs: dict, cu_seqlens, dy, dmu_T=None, dI_T=None):
    """dL/d(input) in fp64 for L = <dy, y> + <dmu_T, mu_T> + <dI_T, I_T> of the
    packed forward. ``inputs`` maps q, k, v, beta, d_t (packed), A, I_prior and
    mu0, I0 ([N, H, dv, dk] or None) to numpy arrays; returns the same keys,
    with zero rows for tokens outside every sequence."""
    from oracle import autograd as ag
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    tok = ("q", "k", "v", "beta", "d_t")
    x = {n: np.asarray(inputs[n], dtype=np.float64) for n in tok + ("A", "I_prior")}
    out = {n: np.zeros_like(x[n]) for n in tok + ("A", "I_prior")}
    H, _, dk = x["q"].shape
    dv = x["v"].shape[-1]
    st = {n: (None if inputs.get(n) is None else np.asarray(inputs[n], dtype=np.float64)) for n in ("mu0", "I0")}
    for n in ("mu0", "I0"):
        if st[n] is not None:
            out[n] = np.zeros((N, H, dv, dk))
    dy = np.asarray(dy, dtype=np.float64)
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        one = {m: x[m][None, :, s0:s1] for m in tok}
        one.update(A=x["A"], I_prior=x["I_prior"],
                   mu0=None if st["mu0"] is None else st["mu0"][n:n + 1],
                   I0=None if st["I0"] is None else st["I0"][n:n + 1])
        g = ag.gradients(one, dy[None, :, s0:s1],
                         None if dmu_T is None else np.asarray(dmu_T, dtype=np.float64)[n:n + 1],
                         None if dI_T is None else np.asarray(dI_T, dtype=np.float64)[n:n + 1])
        for m in tok:
            out[m][:, s0:s1] = g[m][0]
        out["A"] += g["A"]
        out["I_prior"] += g["I_prior"]
        for m in ("mu0", "I0"):
            if st[m] is not None:
                out[m][n] = g[m][0]
    return out
