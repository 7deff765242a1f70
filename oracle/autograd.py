"""ORACLE — test infrastructure only.

Gradients of the Palimpsa recurrence by automatic differentiation in fp64 on
the CPU: ``forward_torch`` is one more plain, token-by-token statement of Eq. (5)
and the readout y_t = mu_t q_t (Bonnet et al., "Learning to Remember, Learn,
and Forget in Attention-Based Models", slide 7 / Eq. (5), slide 4 / Eq. (2)),
written with torch operations so that torch.autograd (a library routine)
differentiates it exactly. ``gradients`` returns dL/d(every input) for
L = <dy, y> + <dmu_T, mu_T> + <dI_T, I_T>.

Pins (tests/test_oracle_pins.py): forward_torch equals the C oracle, and its
gradients equal central finite differences of the C oracle's forward.
"""
from __future__ import annotations

import numpy as np
import torch


def forward_torch(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None):
    """Eq. (5) token by token in torch (fp64 tensors in, fp64 tensors out).
    I_prior is per head [H]. Returns (y, mu_T, I_T)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    Ip = I_prior[None, :, None, None]
    I = Ip.expand(B, H, dv, dk) if I0 is None else I0
    mu = torch.zeros(B, H, dv, dk, dtype=q.dtype) if mu0 is None else mu0
    ys = []
    for t in range(T):
        alpha = torch.exp(-A[None, :] * d_t[:, :, t])[:, :, None, None]
        kt = k[:, :, t, None, :]
        bt = beta[:, :, t, :, None]
        vt = v[:, :, t, :, None]
        I_new = alpha * I + (1.0 - alpha) * Ip + bt * kt ** 2
        mu = alpha * (I / I_new) * mu + (1.0 / I_new) * ((bt * vt) * kt)
        I = I_new
        ys.append(torch.einsum("bhij,bhj->bhi", mu, q[:, :, t, :]))
    y = torch.stack(ys, dim=2) if ys else torch.zeros(B, H, 0, dv, dtype=q.dtype)
    return y, mu, I


NAMES = ("q", "k", "v", "beta", "d_t", "A", "I_prior", "mu0", "I0")


def gradients(inputs: dict, dy, dmu_T=None, dI_T=None):
    """dL/d(input) in fp64 for L = <dy, y> + <dmu_T, mu_T> + <dI_T, I_T>.
    `inputs` maps NAMES to numpy arrays (mu0 / I0 may be None)."""
    t = {n: (None if inputs.get(n) is None else
             torch.tensor(np.asarray(inputs[n], dtype=np.float64), requires_grad=True)) for n in NAMES}
    y, mu, I = forward_torch(*(t[n] for n in NAMES))
    L = (y * torch.tensor(np.asarray(dy, dtype=np.float64))).sum()
    if dmu_T is not None:
        L = L + (mu * torch.tensor(np.asarray(dmu_T, dtype=np.float64))).sum()
    if dI_T is not None:
        L = L + (I * torch.tensor(np.asarray(dI_T, dtype=np.float64))).sum()
    leaves = [n for n in NAMES if t[n] is not None]
    if not L.requires_grad:
        # L reaches no input (an empty sequence with no final-state cotangent, or
        # one whose final state is a constant): every gradient is zero
        return {n: np.zeros(t[n].shape) for n in leaves}
    grads = torch.autograd.grad(L, [t[n] for n in leaves], allow_unused=True)
    out = {}
    for n, gr in zip(leaves, grads):
        out[n] = np.zeros(t[n].shape) if gr is None else gr.detach().numpy()
    return out
