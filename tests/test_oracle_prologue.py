"""Pins for the oracle's fused prologue (``oracle/prologue.py``) and its v* switch.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 10 (Palimpsa-D L2-normalises q and k), slide 11
and reading notes 2.8 (v* = beta (.) v as the kernel input, per-head b_scale,
the Mamba2 limit). Each test is chosen so that a plausible slip in the prologue
(a wrong axis, b_scale applied to the wrong tensor, v* multiplied by beta again,
a sign in an activation) fails it.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import prologue as P
from oracle import reference_np as rnp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _raw_problem(rng, B=1, H=2, T=30, dk=6, dv=4):
    q = rng.standard_normal((B, H, T, dk)) * rng.uniform(0.2, 5.0, (B, H, T, 1))
    k = rng.standard_normal((B, H, T, dk)) * rng.uniform(0.2, 5.0, (B, H, T, 1))
    v = rng.standard_normal((B, H, T, dv))
    b_raw = rng.standard_normal((B, H, T, dv))
    d_raw = rng.normal(-1.0, 1.0, (B, H, T))
    A = rng.uniform(0.1, 1.0, H)
    Ip = rng.uniform(0.5, 2.0, H)
    return q, k, v, b_raw, d_raw, A, Ip


# ---------------------------------------------------------------- activations

def test_sigmoid_printed_value():
    for x, s in _rows("sigmoid_printed.txt"):
        assert abs(float(P.sigmoid(float(x))) - float(s)) < 5e-6


def test_activation_closed_forms():
    x = np.linspace(-30, 30, 241)
    assert P.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    assert P.sigmoid(0.0) == 0.5
    # softplus(x) - softplus(-x) = x ; sigmoid(x) + sigmoid(-x) = 1
    np.testing.assert_allclose(P.softplus(x) - P.softplus(-x), x, atol=1e-13)
    np.testing.assert_allclose(P.sigmoid(x) + P.sigmoid(-x), 1.0, atol=1e-15)
    # library routines for the same functions
    np.testing.assert_allclose(P.softplus(x), np.logaddexp(0.0, x), rtol=1e-14)
    np.testing.assert_allclose(P.sigmoid(x), expit(x), rtol=1e-14)
    # sigmoid is the derivative of softplus (central difference)
    h = 1e-5
    np.testing.assert_allclose((P.softplus(x + h) - P.softplus(x - h)) / (2 * h), P.sigmoid(x), atol=1e-9)
    # tails: no overflow, no lost tail
    assert P.softplus(800.0) == 800.0 and P.softplus(-800.0) == 0.0
    assert P.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert P.sigmoid(-800.0) == 0.0 and P.sigmoid(800.0) == 1.0


def test_l2_normalize_per_token():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 7, 5))
    u = P.l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, rtol=1e-15)
    # invariant to a separate positive scale per token, so the norm runs over d_k only
    c = rng.uniform(0.01, 100.0, (2, 3, 7, 1))
    np.testing.assert_allclose(P.l2_normalize(c * x), u, rtol=1e-14)
    # direction kept
    np.testing.assert_allclose(np.sum(u * x, -1), np.linalg.norm(x, axis=-1), rtol=1e-14)
    assert np.all(P.l2_normalize(np.zeros((4, 8))) == 0.0)


# ---------------------------------------------------------------- the fused forward

def test_v_star_equal_to_beta_times_v_reproduces_the_plain_forward():
    """Slide 11: v* = beta (.) v. Feeding that product as v* must give the plain
    forward's result (the write differs only in where the product is formed)."""
    rng = np.random.default_rng(5)
    q, k, v, b_raw, d_raw, A, Ip = _raw_problem(rng)
    qn, kn, _, beta, d_t = P.apply(q, k, v, b_raw, d_raw, qk_norm=True)
    y, mu, I = oracle.forward(qn, kn, v, beta, d_t, A, Ip)
    ys, mus, Is = oracle.forward(qn, kn, beta * v, beta, d_t, A, Ip, v_star=True)
    np.testing.assert_allclose(ys, y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(mus, mu, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(Is, I)
    # and the step agrees with the forward in v* mode
    mu_s, I_s = np.zeros_like(mu), np.broadcast_to(Ip[None, :, None, None], mu.shape).copy()
    for t in range(q.shape[2]):
        yt, mu_s, I_s = oracle.step(qn[:, :, t], kn[:, :, t], (beta * v)[:, :, t], beta[:, :, t], d_t[:, :, t], A,
                                    Ip, mu_s, I_s, v_star=True)
        np.testing.assert_allclose(yt, ys[:, :, t], rtol=1e-12, atol=1e-14)


def test_v_star_with_vanishing_b_scale_is_the_mamba2_recurrence():
    """Slide 11: with v* as the input and beta -> 0 (b_scale = eps), the mean follows
    mu_t = alpha mu_{t-1} + (v*/I_prior) (x) k_t, the frozen-importance recurrence;
    the distance shrinks in proportion to eps."""
    rng = np.random.default_rng(7)
    q, k, v, b_raw, d_raw, A, Ip = _raw_problem(rng, T=25)
    qn, kn, _, _, d_t = P.apply(q, k, v, b_raw, d_raw, qk_norm=True)
    y_lim, _ = rnp.forward_without_meta(qn, kn, v, np.ones_like(v), d_t, A, Ip)
    errs = []
    for eps in (1e-2, 1e-3, 1e-4):
        y, _, _ = P.forward(q, k, v, b_raw, d_raw, A, Ip, b_scale=np.full(2, eps), qk_norm=True, v_star=True)
        errs.append(np.linalg.norm(y - y_lim) / np.linalg.norm(y_lim))
    assert errs[-1] < 1e-3
    for a, b in zip(errs, errs[1:]):
        assert 7.0 < a / b < 13.0, errs


def test_b_scale_scales_the_importance_gate():
    """b_scale multiplies beta: b_scale = c with I_prior and I_0 scaled by c leaves
    mu and y as with b_scale = 1 and scales I by c (Eq. 5's scale invariance)."""
    rng = np.random.default_rng(9)
    q, k, v, b_raw, d_raw, A, Ip = _raw_problem(rng)
    I0 = rng.uniform(0.5, 3.0, (1, 2, 4, 6))
    mu0 = rng.standard_normal((1, 2, 4, 6))
    c = np.array([0.3, 2.5])
    y, mu, I = P.forward(q, k, v, b_raw, d_raw, A, Ip, mu0=mu0, I0=I0, qk_norm=True)
    yc, muc, Ic = P.forward(q, k, v, b_raw, d_raw, A, c * Ip, b_scale=c, mu0=mu0, I0=c[None, :, None, None] * I0,
                            qk_norm=True)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(muc, mu, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(Ic, c[None, :, None, None] * I, rtol=1e-12)


def test_qk_norm_makes_the_forward_blind_to_per_token_scales():
    rng = np.random.default_rng(11)
    q, k, v, b_raw, d_raw, A, Ip = _raw_problem(rng)
    y, mu, I = P.forward(q, k, v, b_raw, d_raw, A, Ip, qk_norm=True)
    cq = rng.uniform(0.05, 20.0, q.shape[:-1] + (1,))
    ck = rng.uniform(0.05, 20.0, k.shape[:-1] + (1,))
    y2, mu2, I2 = P.forward(cq * q, ck * k, v, b_raw, d_raw, A, Ip, qk_norm=True)
    np.testing.assert_allclose(y2, y, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(I2, I, rtol=1e-12)
    # without the norm, the raw scale reaches I through k^2
    _, _, I3 = P.forward(cq * q, ck * k, v, b_raw, d_raw, A, Ip, qk_norm=False)
    assert np.max(np.abs(I3 - I)) > 1e-3


def test_gate_domain_after_the_prologue():
    """Any real raw input lands in the recurrence's domain: d_t > 0, 0 < beta <= b_scale."""
    rng = np.random.default_rng(13)
    q, k, v, b_raw, d_raw, A, Ip = _raw_problem(rng)
    b_raw = b_raw * 30.0
    d_raw = d_raw * 30.0
    _, _, _, beta, d_t = P.apply(q, k, v, b_raw, d_raw, b_scale=np.array([0.1, 1.0]))
    assert np.all(d_t >= 0.0) and np.all(beta >= 0.0)
    assert np.all(beta[:, 0] <= 0.1) and np.all(beta[:, 1] <= 1.0)
