"""ORACLE — test infrastructure only.

NumPy fp64 statements of the Palimpsa recurrence, independent of the C oracle
in ``palimpsa_oracle.c`` (they share no code) and of the CUDA library. Only the
tests, the smoke check and the benchmark's CPU-baseline leg may import this.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — its slide deck and its Chinese reading notes.

* ``forward_mu_form``: Eq. (5) in its mean/precision form (slide 7; reading
  notes section 2.5), token by token, every row and key index at once.
* ``forward_natural_chunked``: the natural-parameter form (slide 9, App. A.12;
  reading notes section 2.6) evaluated chunk by chunk: inside a chunk every
  token's (M_t, Ibar_t) is written in closed form as a decayed sum over the
  chunk's writes (the "parallel scan within the chunk"), and the end state is
  carried to the next chunk in sequence.
* ``forward_without_meta``: the same recurrence with the importance frozen at
  I_prior (slide 10's "without Meta" ablation; slide 11's Mamba2 limit),
  token by token.
* ``forward_full_gaussian``: the coupled Gaussian posterior that Eq. (5)
  approximates (slide 25, App. A.3-A.5; reading notes section 2.5), with a full
  dk x dk precision matrix per value row. Used only on tiny inputs.

Array layouts follow the C oracle: q, k [B, H, T, dk]; v, beta [B, H, T, dv];
d_t [B, H, T]; A [H]; I_prior [H] (or [H, dv, dk]); states [B, H, dv, dk];
y [B, H, T, dv].
"""
from __future__ import annotations

import numpy as np


def _prior_grid(I_prior, H, dv, dk):
    """I_prior as a [H, dv, dk] array (per-head scalar broadcast over states)."""
    Ip = np.asarray(I_prior, dtype=np.float64)
    if Ip.ndim == 1:
        return np.broadcast_to(Ip[:, None, None], (H, dv, dk)).copy()
    return Ip.reshape(H, dv, dk).copy()


def _initial_state(mu0, I0, Ipg, B):
    H, dv, dk = Ipg.shape
    mu = np.zeros((B, H, dv, dk)) if mu0 is None else np.array(mu0, dtype=np.float64)
    I = np.broadcast_to(Ipg, (B, H, dv, dk)).copy() if I0 is None else np.array(I0, dtype=np.float64)
    return mu, I


def forward_mu_form(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None):
    """Eq. (5) and the readout y_t = mu_t q_t, one token at a time.

    alpha_t = exp(-A d_t) (slide 5); I_t = alpha I_{t-1} + (1 - alpha) I_prior
    + beta (x) k^2; mu_t = alpha (I_{t-1}/I_t) mu_{t-1} + (1/I_t)((beta v) (x) k)
    (slide 7); the read uses the updated mean (slide 4, Eq. 2).
    Returns (y, mu_T, I_T).
    """
    q, k, v, beta, d_t = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, d_t))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Ipg = _prior_grid(I_prior, H, dv, dk)
    mu, I = _initial_state(mu0, I0, Ipg, B)
    A = np.asarray(A, dtype=np.float64)
    y = np.zeros((B, H, T, dv))
    for t in range(T):
        alpha = np.exp(-A[None, :] * d_t[:, :, t])[:, :, None, None]          # [B,H,1,1]
        kt = k[:, :, t, None, :]                                               # [B,H,1,dk]
        bt = beta[:, :, t, :, None]                                            # [B,H,dv,1]
        vt = v[:, :, t, :, None]
        I_new = alpha * I + (1.0 - alpha) * Ipg[None] + bt * kt ** 2
        mu = alpha * (I / I_new) * mu + (1.0 / I_new) * ((bt * vt) * kt)
        I = I_new
        y[:, :, t, :] = np.einsum("bhij,bhj->bhi", mu, q[:, :, t, :])
    return y, mu, I


def forward_natural_chunked(q, k, v, beta, d_t, A, I_prior, chunk, mu0=None, I0=None):
    """Natural parameters M = I (.) mu and Ibar = I - I_prior (slide 9, App. A.12).

    M_t = alpha_t M_{t-1} + (beta (.) v) (x) k,  Ibar_t = alpha_t Ibar_{t-1} + beta (x) k^2,
    y_t = (M_t / (I_prior + Ibar_t)) q_t.
    Inside a chunk starting at s0, with G[t, s] = prod_{u=s+1..t} alpha_u
    (products, never quotients of cumulative products):
    M_t = G[t, s0-1] M_{s0-1} + sum_{s0<=s<=t} G[t, s] (beta_s v_s) (x) k_s,
    and likewise for Ibar. The chunk's last state is carried to the next chunk.
    Returns (y, mu_T, I_T).
    """
    q, k, v, beta, d_t = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, d_t))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Ipg = _prior_grid(I_prior, H, dv, dk)
    mu, I = _initial_state(mu0, I0, Ipg, B)
    M = I * mu
    Ib = I - Ipg[None]
    alpha_all = np.exp(-np.asarray(A, dtype=np.float64)[None, :, None] * d_t)   # [B,H,T]
    y = np.zeros((B, H, T, dv))
    for s0 in range(0, T, chunk):
        s1 = min(T, s0 + chunk)
        C = s1 - s0
        al = alpha_all[:, :, s0:s1]                                           # [B,H,C]
        # G[b,h,t,s] = prod_{u=s+1..t} alpha_u for s <= t (t, s chunk-local), 0 above.
        G = np.zeros((B, H, C, C))
        for t in range(C):
            G[:, :, t, t] = 1.0
            for s in range(t - 1, -1, -1):
                G[:, :, t, s] = G[:, :, t, s + 1] * al[:, :, s + 1]
        # decay from the carried state: prod_{u=s0..t} alpha_u
        g0 = np.zeros((B, H, C))
        g0[:, :, 0] = al[:, :, 0]
        for t in range(1, C):
            g0[:, :, t] = g0[:, :, t - 1] * al[:, :, t]
        bv = beta[:, :, s0:s1, :] * v[:, :, s0:s1, :]                          # [B,H,C,dv]
        kc = k[:, :, s0:s1, :]
        Mt = g0[..., None, None] * M[:, :, None] + np.einsum("bhts,bhsi,bhsj->bhtij", G, bv, kc)
        Ibt = g0[..., None, None] * Ib[:, :, None] + np.einsum(
            "bhts,bhsi,bhsj->bhtij", G, beta[:, :, s0:s1, :], kc ** 2)
        mu_t = Mt / (Ipg[None, :, None] + Ibt)
        y[:, :, s0:s1, :] = np.einsum("bhtij,bhtj->bhti", mu_t, q[:, :, s0:s1, :])
        M = Mt[:, :, -1]
        Ib = Ibt[:, :, -1]
    I_T = Ipg[None] + Ib
    return y, M / I_T, I_T


def forward_full_gaussian(q, k, v, beta, d_t, A, I_prior, P0=None, mu0=None):
    """Coupled Gaussian posterior per value row (slide 25, App. A.3-A.5).

    P_t = alpha P_{t-1} + (1 - alpha) P_prior + beta_i k k^T, P_prior = I_prior Id,
    mu_t = P_t^{-1} [alpha P_{t-1} mu_{t-1} + beta_i v_i k]; y_t = mu_t q_t.
    I_prior must be a per-head scalar [H]. P0 [B,H,dv,dk,dk] defaults to
    P_prior; mu0 [B,H,dv,dk] defaults to 0. Returns (y, mu_T, P_T).
    """
    q, k, v, beta, d_t = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, d_t))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Ip = np.asarray(I_prior, dtype=np.float64)
    eye = np.eye(dk)
    P = np.empty((B, H, dv, dk, dk))
    for h in range(H):
        P[:, h] = Ip[h] * eye
    if P0 is not None:
        P = np.array(P0, dtype=np.float64)
    mu = np.zeros((B, H, dv, dk)) if mu0 is None else np.array(mu0, dtype=np.float64)
    y = np.zeros((B, H, T, dv))
    for b in range(B):
        for h in range(H):
            Pprior = Ip[h] * eye
            for t in range(T):
                alpha = np.exp(-A[h] * d_t[b, h, t])
                kt = k[b, h, t]
                for i in range(dv):
                    Pn = alpha * P[b, h, i] + (1 - alpha) * Pprior + beta[b, h, t, i] * np.outer(kt, kt)
                    rhs = alpha * P[b, h, i] @ mu[b, h, i] + beta[b, h, t, i] * v[b, h, t, i] * kt
                    mu[b, h, i] = np.linalg.solve(Pn, rhs)
                    P[b, h, i] = Pn
                y[b, h, t] = mu[b, h] @ q[b, h, t]
    return y, mu, P


def forward_without_meta(q, k, v, beta, d_t, A, I_prior, mu0=None):
    """Importance frozen at the prior (slide 11): mu_t = alpha_t mu_{t-1}
    + ((beta_t v_t) / I_prior) (x) k_t, y_t = mu_t q_t. I_prior is per head [H].
    Returns (y, mu_T)."""
    q, k, v, beta, d_t = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, d_t))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Ip = np.asarray(I_prior, dtype=np.float64)[None, :, None, None]
    mu = np.zeros((B, H, dv, dk)) if mu0 is None else np.array(mu0, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    y = np.zeros((B, H, T, dv))
    for t in range(T):
        alpha = np.exp(-A[None, :] * d_t[:, :, t])[:, :, None, None]
        mu = alpha * mu + ((beta[:, :, t, :, None] * v[:, :, t, :, None]) / Ip) * k[:, :, t, None, :]
        y[:, :, t, :] = np.einsum("bhij,bhj->bhi", mu, q[:, :, t, :])
    return y, mu
