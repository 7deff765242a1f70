"""Pins for the fp64 oracle: values and identities that the pages and the
mathematics fix, chosen so that a dropped term, a flipped sign, a wrong index
or a swapped operand in the oracle fails at least one of them.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" (slide deck and Chinese reading notes).
"""
import math
import os

import numpy as np
import pytest
from scipy.optimize import minimize

import oracle
from oracle import reference_np as rnp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _random_problem(rng, B=1, H=2, T=40, dk=6, dv=5, unit_keys=True):
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T, dv))))
    d_t = np.log1p(np.exp(rng.standard_normal((B, H, T))))
    A = rng.uniform(0.1, 1.0, H)
    I_prior = rng.uniform(0.5, 2.0, H)
    return q, k, v, beta, d_t, A, I_prior


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- printed examples

@pytest.mark.parametrize("impl", ["c", "numpy"])
def test_slide8_scalar_example(impl):
    """Slide 8 table: a confident state (I_{t-1}=9) keeps more of its old mean."""
    for I_prev, I_new, mu_new in _read_rows("slide8_scalar_example.txt"):
        I_prev, I_new, mu_new = float(I_prev), float(I_new), float(mu_new)
        args = dict(q=np.ones((1, 1, 1, 1)), k=np.ones((1, 1, 1, 1)), v=np.zeros((1, 1, 1, 1)),
                    beta=np.ones((1, 1, 1, 1)), d_t=np.full((1, 1, 1), -math.log(0.9)),
                    A=np.ones(1), I_prior=np.ones(1))
        mu0 = np.ones((1, 1, 1, 1))
        I0 = np.full((1, 1, 1, 1), I_prev)
        if impl == "c":
            y, muT, IT = oracle.forward(**args, mu0=mu0, I0=I0)
        else:
            y, muT, IT = rnp.forward_mu_form(**args, mu0=mu0, I0=I0)
        assert IT[0, 0, 0, 0] == pytest.approx(I_new, abs=1e-12)
        assert muT[0, 0, 0, 0] == pytest.approx(mu_new, abs=5e-5)      # printed to 4 decimals
        assert y[0, 0, 0, 0] == pytest.approx(muT[0, 0, 0, 0], abs=1e-15)  # q = 1 reads the new mean


def test_slide25_full_vs_diagonal():
    """Slide 25: the coupled posterior gives mu = (1/3, 1/3); Palimpsa's diagonal gives (1/2, 1/2)."""
    rows = {r[0]: [float(x) for x in r[1:]] for r in _read_rows("slide25_full_vs_diag.txt")}
    for alpha in (0.3, 0.9, 1.0):
        d = -math.log(alpha)
        args = dict(q=np.array([[[[1.0, 0.0]]]]), k=np.ones((1, 1, 1, 2)), v=np.ones((1, 1, 1, 1)),
                    beta=np.ones((1, 1, 1, 1)), d_t=np.full((1, 1, 1), d), A=np.ones(1),
                    I_prior=np.ones(1))
        _, mu_d, I_d = oracle.forward(**args)
        np.testing.assert_allclose(mu_d[0, 0, 0], rows["mu_diag"], atol=1e-15)
        np.testing.assert_allclose(I_d[0, 0, 0], [2.0, 2.0], atol=1e-15)
        _, mu_f, P_f = rnp.forward_full_gaussian(**args)
        np.testing.assert_allclose(P_f[0, 0, 0].ravel(), rows["P_full"], atol=1e-15)
        np.testing.assert_allclose(mu_f[0, 0, 0], rows["mu_full"], atol=1e-15)


# ---------------------------------------------------------------- exact special cases

@pytest.mark.parametrize("seed", [0, 1])
def test_axis_aligned_keys_equal_full_gaussian(seed):
    """With one-hot keys k = c e_j the coupled update never creates off-diagonal
    precision, so Eq. (5) is the exact posterior (App. A.5): the oracle must equal
    the full-Gaussian brute force over a long random sequence."""
    rng = _rng(seed)
    B, H, T, dk, dv = 1, 2, 60, 4, 3
    q, _, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv)
    k = np.zeros((B, H, T, dk))
    idx = rng.integers(0, dk, size=(B, H, T))
    mag = rng.uniform(-2.0, 2.0, size=(B, H, T))
    np.put_along_axis(k, idx[..., None], mag[..., None], axis=-1)
    I0 = rng.uniform(0.3, 5.0, (B, H, dv, dk))
    mu0 = rng.standard_normal((B, H, dv, dk))
    P0 = np.zeros((B, H, dv, dk, dk))
    for j in range(dk):
        P0[..., j, j] = I0[..., j]
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    yf, muf, Pf = rnp.forward_full_gaussian(q, k, v, beta, d_t, A, I_prior, P0=P0, mu0=mu0)
    np.testing.assert_allclose(y, yf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(muT, muf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(IT, np.diagonal(Pf, axis1=-2, axis2=-1), rtol=1e-12)
    off = Pf - np.einsum("...ij,ij->...ij", Pf, np.eye(dk))
    assert np.abs(off).max() == 0.0


def test_scalar_key_equals_full_gaussian():
    """d_k = 1: the full and diagonal posteriors coincide for arbitrary keys."""
    rng = _rng(7)
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, 1, 2, 80, 1, 4, unit_keys=False)
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior)
    yf, muf, Pf = rnp.forward_full_gaussian(q, k, v, beta, d_t, A, I_prior)
    np.testing.assert_allclose(y, yf, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(IT[..., 0], Pf[..., 0, 0], rtol=1e-12)


def _free_energy_argmin(mu_prev, P_prev, alpha, Ip, b, v, k, diagonal):
    """Minimise the per-row free energy of Eq. (3) (slide 6) numerically.

    F(mu) = b/2 (fit) + (1-alpha) Ip/2 |mu|^2 + alpha/2 (mu - mu_prev)^T P_prev (mu - mu_prev),
    where the fit term is (mu.k - v)^2 for the coupled posterior, and becomes
    sum_j k_j^2 mu_j^2 - 2 v k.mu + v^2 when k k^T is replaced by diag(k^2)
    (the diagonal approximation of App. A.5)."""
    def F(mu):
        if diagonal:
            fit = np.sum(k ** 2 * mu ** 2) - 2 * v * np.dot(k, mu) + v * v
        else:
            fit = (np.dot(mu, k) - v) ** 2
        dmu = mu - mu_prev
        return 0.5 * b * fit + 0.5 * (1 - alpha) * Ip * np.dot(mu, mu) + 0.5 * alpha * dmu @ P_prev @ dmu

    res = minimize(F, np.zeros_like(mu_prev), method="BFGS", options={"gtol": 1e-12, "maxiter": 10000})
    return res.x


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_eq5_is_argmin_of_eq3_with_diagonal_metric(seed):
    """One step of Eq. (5) is the minimiser of Eq. (3) with k k^T -> diag(k^2) and a
    diagonal history precision; the coupled minimiser is the full-Gaussian step."""
    rng = _rng(seed)
    dk = 4
    mu_prev = rng.standard_normal(dk)
    I_prev = rng.uniform(0.5, 4.0, dk)
    alpha, Ip, b, v = 0.8, 1.3, 0.7, 1.9
    k = rng.standard_normal(dk)
    args = dict(q=np.ones((1, 1, 1, dk)), k=k.reshape(1, 1, 1, dk), v=np.full((1, 1, 1, 1), v),
                beta=np.full((1, 1, 1, 1), b), d_t=np.full((1, 1, 1), -math.log(alpha)),
                A=np.ones(1), I_prior=np.full(1, Ip))
    _, muT, IT = oracle.forward(**args, mu0=mu_prev.reshape(1, 1, 1, dk), I0=I_prev.reshape(1, 1, 1, dk))
    target = _free_energy_argmin(mu_prev, np.diag(I_prev), alpha, Ip, b, v, k, diagonal=True)
    np.testing.assert_allclose(muT[0, 0, 0], target, atol=1e-6)
    _, muf, _ = rnp.forward_full_gaussian(**args, P0=np.diag(I_prev).reshape(1, 1, 1, dk, dk),
                                          mu0=mu_prev.reshape(1, 1, 1, dk))
    target_full = _free_energy_argmin(mu_prev, np.diag(I_prev), alpha, Ip, b, v, k, diagonal=False)
    np.testing.assert_allclose(muf[0, 0, 0], target_full, atol=1e-6)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("impl", ["c", "numpy"])
def test_discount_without_evidence(impl):
    """beta = 0 (slide 8, reading notes 2.5): I_n - I_prior = (prod alpha)(I_0 - I_prior)
    and the content decays as mu_n = (prod alpha) I_0 mu_0 / I_n."""
    rng = _rng(11)
    B, H, T, dk, dv = 2, 3, 30, 5, 4
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv)
    beta[:] = 0.0
    I0 = rng.uniform(0.2, 6.0, (B, H, dv, dk))
    mu0 = rng.standard_normal((B, H, dv, dk))
    f = oracle.forward if impl == "c" else rnp.forward_mu_form
    y, muT, IT = f(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    G = np.exp(-np.sum(A[None, :, None] * d_t, axis=-1))[..., None, None]     # prod of alpha
    Ip = I_prior[None, :, None, None]
    np.testing.assert_allclose(IT - Ip, G * (I0 - Ip), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(muT, G * I0 * mu0 / IT, rtol=1e-11, atol=1e-14)


def test_stationary_precision_closed_form():
    """Constant alpha, beta, k (slide 27): I_t = I_prior + beta k^2 (1 - alpha^t)/(1 - alpha)
    + alpha^t (I_0 - I_prior) at every t, hence I_inf = I_prior + N beta k^2."""
    B, H, dk, dv, T = 1, 1, 3, 2, 400
    alpha, Ip = 0.95, 1.7
    kk = np.array([0.7, -1.3, 0.2])
    bb = np.array([0.4, 0.9])
    I0 = np.full((B, H, dv, dk), 3.0)
    I = I0.copy()
    mu = np.zeros_like(I)
    for t in range(1, T + 1):
        _, mu, I = oracle.step(np.ones((1, 1, dk)), kk.reshape(1, 1, dk), np.ones((1, 1, dv)),
                               bb.reshape(1, 1, dv), np.full((1, 1), -math.log(alpha)), np.ones(1),
                               np.full(1, Ip), mu, I)
        expect = Ip + np.outer(bb, kk ** 2) * (1 - alpha ** t) / (1 - alpha) + alpha ** t * (I0[0, 0] - Ip)
        np.testing.assert_allclose(I[0, 0], expect, rtol=1e-12)
    N = 1.0 / (1.0 - alpha)
    np.testing.assert_allclose(I[0, 0], Ip + N * np.outer(bb, kk ** 2), rtol=1e-7)


def _scalar_decay_readout(q, k, vstar, d_t, A, I_prior):
    """Mamba2 / scalar-decay linear attention written as an explicit sum:
    y_t = sum_{s<=t} (prod_{u=s+1..t} alpha_u) (v*_s / I_prior) (k_s . q_t)."""
    B, H, T, dk = q.shape
    dv = vstar.shape[-1]
    alpha = np.exp(-A[None, :, None] * d_t)
    y = np.zeros((B, H, T, dv))
    for t in range(T):
        w = np.ones((B, H))
        for s in range(t, -1, -1):
            score = np.einsum("bhj,bhj->bh", k[:, :, s], q[:, :, t])
            y[:, :, t] += (w * score)[..., None] * vstar[:, :, s] / I_prior[None, :, None]
            w = w * alpha[:, :, s]
    return y


def test_mamba2_limit():
    """Slide 11 / reading notes 2.8: for small excess precision, with v* = beta v held
    fixed and beta = eps -> 0, the mean follows mu_t = alpha mu_{t-1} + (v*/I_prior) (x) k.
    The oracle's distance to that limit must shrink in proportion to eps."""
    rng = _rng(21)
    B, H, T, dk, dv = 1, 2, 25, 6, 3
    q, k, _, _, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv)
    vstar = rng.standard_normal((B, H, T, dv))
    y_lim = _scalar_decay_readout(q, k, vstar, d_t, A, I_prior)
    errs = []
    for eps in (1e-2, 1e-3, 1e-4):
        beta = np.full((B, H, T, dv), eps)
        y, _, IT = oracle.forward(q, k, vstar / eps, beta, d_t, A, I_prior)
        errs.append(np.linalg.norm(y - y_lim) / np.linalg.norm(y_lim))
    assert errs[-1] < 1e-3
    for a, b in zip(errs, errs[1:]):
        assert 7.0 < a / b < 13.0, errs


# ---------------------------------------------------------------- invariants

def test_positivity_of_precision():
    """I stays >= min(I_0, I_prior) > 0 (alpha in (0,1], beta >= 0), and the excess
    precision I - I_prior stays >= 0 when I_0 >= I_prior."""
    rng = _rng(31)
    B, H, T, dk, dv = 1, 2, 200, 5, 4
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv, unit_keys=False)
    I0 = I_prior[None, :, None, None] * rng.uniform(0.1, 3.0, (B, H, dv, dk))
    mu = rng.standard_normal((B, H, dv, dk))
    I = I0.copy()
    lo = np.minimum(I0, I_prior[None, :, None, None])
    for t in range(T):
        _, mu, I = oracle.step(q[:, :, t], k[:, :, t], v[:, :, t], beta[:, :, t], d_t[:, :, t], A,
                               I_prior, mu, I)
        assert np.all(I >= lo * (1 - 1e-15))
    I0b = I_prior[None, :, None, None] + rng.uniform(0.0, 2.0, (B, H, dv, dk))
    _, _, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, I0=I0b, mu0=np.zeros_like(I0b))
    assert np.all(IT - I_prior[None, :, None, None] >= 0)


def test_row_independence():
    """Each value row sees only its own beta_i and v_i: running rows separately
    reproduces the full run."""
    rng = _rng(41)
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, 2, 2, 30, 5, 4)
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior)
    for i in range(v.shape[-1]):
        yi, mui, Ii = oracle.forward(q, k, v[..., i:i + 1], beta[..., i:i + 1], d_t, A, I_prior)
        np.testing.assert_array_equal(yi[..., 0], y[..., i])
        np.testing.assert_array_equal(mui[:, :, 0], muT[:, :, i])
        np.testing.assert_array_equal(Ii[:, :, 0], IT[:, :, i])


def test_linearity_in_v():
    """With mu_0 = 0, I does not depend on v and y is linear in v."""
    rng = _rng(51)
    q, k, v1, beta, d_t, A, I_prior = _random_problem(rng, 1, 2, 40, 6, 3)
    v2 = rng.standard_normal(v1.shape)
    a, b = 0.7, -2.3
    y1, _, I1 = oracle.forward(q, k, v1, beta, d_t, A, I_prior)
    y2, _, I2 = oracle.forward(q, k, v2, beta, d_t, A, I_prior)
    y3, _, I3 = oracle.forward(q, k, a * v1 + b * v2, beta, d_t, A, I_prior)
    np.testing.assert_array_equal(I1, I2)
    np.testing.assert_allclose(y3, a * y1 + b * y2, rtol=1e-10, atol=1e-12)


def test_prior_scale_invariance():
    """Scaling beta, I_prior and I_0 by c > 0 leaves mu and y unchanged and scales I by c
    (derived from Eq. 5: every term of I scales by c and mu is a ratio)."""
    rng = _rng(61)
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, 1, 2, 50, 5, 4)
    I0 = rng.uniform(0.5, 3.0, (1, 2, 4, 5))
    mu0 = rng.standard_normal((1, 2, 4, 5))
    c = 3.7
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    yc, muc, Ic = oracle.forward(q, k, v, c * beta, d_t, A, c * I_prior, mu0=mu0, I0=c * I0)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(muc, muT, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(Ic, c * IT, rtol=1e-12)


def test_without_meta_matches_the_explicit_decayed_sum_and_the_limit():
    """The frozen-importance oracle (slide 10 / slide 11) equals the separately written
    scalar-decay sum, and Palimpsa's oracle approaches it in the Mamba2 limit."""
    rng = _rng(23)
    B, H, T, dk, dv = 1, 2, 30, 5, 3
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv)
    y, muT = rnp.forward_without_meta(q, k, v, beta, d_t, A, I_prior)
    y_sum = _scalar_decay_readout(q, k, beta * v, d_t, A, I_prior)
    np.testing.assert_allclose(y, y_sum, rtol=1e-11, atol=1e-13)
    eps = 1e-6
    y_lim, _, _ = oracle.forward(q, k, beta * v / eps, np.full_like(beta, eps), d_t, A, I_prior)
    assert np.linalg.norm(y_lim - y) / np.linalg.norm(y) < 1e-4
    # continuation from a nonzero mean
    mu0 = rng.standard_normal((B, H, dv, dk))
    y1, m1 = rnp.forward_without_meta(q[:, :, :11], k[:, :, :11], v[:, :, :11], beta[:, :, :11], d_t[:, :, :11], A,
                                      I_prior, mu0)
    y2, m2 = rnp.forward_without_meta(q[:, :, 11:], k[:, :, 11:], v[:, :, 11:], beta[:, :, 11:], d_t[:, :, 11:], A,
                                      I_prior, m1)
    yf, mf = rnp.forward_without_meta(q, k, v, beta, d_t, A, I_prior, mu0)
    np.testing.assert_allclose(np.concatenate([y1, y2], 2), yf, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(m2, mf, rtol=1e-12, atol=1e-14)


def test_autograd_oracle_forward_equals_the_c_oracle():
    from oracle import autograd as ag
    import torch
    rng = _rng(81)
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, 2, 2, 20, 5, 3)
    mu0 = rng.standard_normal((2, 2, 3, 5))
    I0 = rng.uniform(0.5, 3.0, (2, 2, 3, 5))
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    tt = [torch.tensor(x) for x in (q, k, v, beta, d_t, A, I_prior, mu0, I0)]
    y2, mu2, I2 = ag.forward_torch(*tt)
    np.testing.assert_allclose(y2.numpy(), y, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(mu2.numpy(), muT, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(I2.numpy(), IT, rtol=1e-13)


@pytest.mark.parametrize("with_state", [False, True])
def test_autograd_gradients_equal_finite_differences_of_the_c_oracle(with_state):
    """The gradient oracle is pinned to central differences of a different
    implementation (the C oracle), on a tiny problem, for every input."""
    from oracle import autograd as ag
    rng = _rng(82 + with_state)
    B, H, T, dk, dv = 1, 2, 6, 3, 2
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, T, dk, dv, unit_keys=False)
    inp = dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=I_prior, mu0=None, I0=None)
    if with_state:
        inp["mu0"] = rng.standard_normal((B, H, dv, dk))
        inp["I0"] = rng.uniform(0.5, 2.0, (B, H, dv, dk))
    dy = rng.standard_normal((B, H, T, dv))
    dmu = rng.standard_normal((B, H, dv, dk))
    dI = rng.standard_normal((B, H, dv, dk))
    g = ag.gradients(inp, dy, dmu, dI)

    def loss(d):
        y, muT, IT = oracle.forward(d["q"], d["k"], d["v"], d["beta"], d["d_t"], d["A"], d["I_prior"],
                                    mu0=d["mu0"], I0=d["I0"])
        return float(np.sum(y * dy) + np.sum(muT * dmu) + np.sum(IT * dI))

    h = 1e-6
    for name, arr in inp.items():
        if arr is None:
            continue
        fd = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            dp = {n: (None if a_ is None else np.array(a_, dtype=np.float64)) for n, a_ in inp.items()}
            dm = {n: (None if a_ is None else np.array(a_, dtype=np.float64)) for n, a_ in inp.items()}
            dp[name][idx] += h
            dm[name][idx] -= h
            fd[idx] = (loss(dp) - loss(dm)) / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=2e-6, atol=2e-7, err_msg=name)


def test_autograd_gradients_of_an_empty_sequence():
    """T = 0: the final state is the initial one, so dmu0 = dmu_T and dI0 = dI_T
    exactly (mu_T = mu0, I_T = I0); with no final-state cotangent the loss is a
    constant and every gradient is zero, A and I_prior included."""
    from oracle import autograd as ag
    rng = _rng(90)
    B, H, dk, dv = 1, 2, 3, 2
    q, k, v, beta, d_t, A, I_prior = _random_problem(rng, B, H, 0, dk, dv, unit_keys=False)
    inp = dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=I_prior,
               mu0=rng.standard_normal((B, H, dv, dk)), I0=rng.uniform(0.5, 2.0, (B, H, dv, dk)))
    dmu = rng.standard_normal((B, H, dv, dk))
    dI = rng.standard_normal((B, H, dv, dk))
    g = ag.gradients(inp, np.zeros((B, H, 0, dv)), dmu, dI)
    np.testing.assert_array_equal(g["mu0"], dmu)
    np.testing.assert_array_equal(g["I0"], dI)
    assert not g["A"].any() and not g["I_prior"].any()
    g0 = ag.gradients(inp, np.zeros((B, H, 0, dv)))
    for name in ("mu0", "I0", "A", "I_prior"):
        assert not g0[name].any(), name
