"""Pins for the oracle's packed variable-length forward (``oracle/varlen.py``).

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 7 / Eq. (5) per sequence, slide 9 (the state
carried along one sequence). Each pin ties the packed layout to the dense,
already pinned oracle in a way a wrong offset, a swapped state index or a
leaked state between sequences would break."""
import numpy as np

import oracle
from oracle import varlen as ovl


def _packed(rng, H, lengths, dk, dv, gap=0):
    total = sum(lengths) + gap
    q = rng.standard_normal((H, total, dk))
    k = rng.standard_normal((H, total, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((H, total, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((H, total, dv))))
    d_t = np.log1p(np.exp(rng.standard_normal((H, total))))
    A = rng.uniform(0.1, 1.0, H)
    Ip = rng.uniform(0.5, 2.0, H)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, beta, d_t, A, Ip, cu


def test_equal_lengths_equal_the_dense_batch():
    rng = np.random.default_rng(1)
    B, H, T, dk, dv = 3, 2, 17, 6, 4
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, [T] * B, dk, dv)
    y, muT, IT = ovl.forward(q, k, v, beta, d_t, A, Ip, cu)
    dense = lambda x: x.reshape((H, B, T) + x.shape[2:]).swapaxes(0, 1)   # [H, B*T, .] -> [B, H, T, .]
    yd, mud, Id = oracle.forward(dense(q), dense(k), dense(v), dense(beta), dense(d_t), A, Ip)
    np.testing.assert_array_equal(dense(y), yd)
    np.testing.assert_array_equal(muT, mud)
    np.testing.assert_array_equal(IT, Id)


def test_state_handed_across_sequences_equals_one_long_run():
    rng = np.random.default_rng(2)
    H, dk, dv = 2, 5, 3
    lengths = [9, 1, 30, 14]
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, lengths, dk, dv)
    y_long, mu_long, I_long = oracle.forward(q[None], k[None], v[None], beta[None], d_t[None], A, Ip)
    mu0 = np.zeros((1, H, dv, dk))
    I0 = np.broadcast_to(Ip[None, :, None, None], (1, H, dv, dk)).copy()
    for n in range(len(lengths)):
        y, mu, I = ovl.forward(q, k, v, beta, d_t, A, Ip, cu[n:n + 2], mu0=mu0, I0=I0)
        s0, s1 = cu[n], cu[n + 1]
        np.testing.assert_allclose(y[:, s0:s1], y_long[0, :, s0:s1], rtol=1e-12, atol=1e-14)
        mu0, I0 = mu, I
    np.testing.assert_allclose(mu0[0], mu_long[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(I0[0], I_long[0], rtol=1e-12)


def test_empty_sequences_and_unused_tokens():
    rng = np.random.default_rng(3)
    H, dk, dv = 2, 4, 3
    lengths = [0, 12, 0, 5]
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, lengths, dk, dv, gap=6)
    N = len(lengths)
    mu0 = rng.standard_normal((N, H, dv, dk))
    I0 = rng.uniform(0.5, 3.0, (N, H, dv, dk))
    y, muT, IT = ovl.forward(q, k, v, beta, d_t, A, Ip, cu, mu0=mu0, I0=I0)
    for n in (0, 2):
        np.testing.assert_array_equal(muT[n], mu0[n])
        np.testing.assert_array_equal(IT[n], I0[n])
    assert np.all(y[:, cu[-1]:] == 0.0)
    # the unused tail is never read
    q2, k2 = q.copy(), k.copy()
    q2[:, cu[-1]:] = np.nan
    k2[:, cu[-1]:] = np.nan
    y2, mu2, I2 = ovl.forward(q2, k2, v, beta, d_t, A, Ip, cu, mu0=mu0, I0=I0)
    np.testing.assert_array_equal(y2[:, :cu[-1]], y[:, :cu[-1]])
    np.testing.assert_array_equal(mu2, muT)
    # a sequence does not see its neighbours: perturbing sequence 3 leaves sequence 1 alone
    v3 = v.copy()
    v3[:, cu[3]:cu[4]] += 1.0
    y3, mu3, _ = ovl.forward(q, k, v3, beta, d_t, A, Ip, cu, mu0=mu0, I0=I0)
    np.testing.assert_array_equal(y3[:, cu[1]:cu[2]], y[:, cu[1]:cu[2]])
    np.testing.assert_array_equal(mu3[1], muT[1])
    assert not np.allclose(mu3[3], muT[3])


def _packed_loss(x, cu, dy, dmu, dI):
    y, muT, IT = ovl.forward(x["q"], x["k"], x["v"], x["beta"], x["d_t"], x["A"], x["I_prior"], cu,
                             mu0=x["mu0"], I0=x["I0"])
    return float((y * dy).sum() + (muT * dmu).sum() + (IT * dI).sum())


def test_packed_gradients_equal_finite_differences_of_the_packed_forward():
    """Every input's gradient from ovl.gradients (per-sequence autograd, A and
    I_prior summed) against central differences of the packed C-oracle forward:
    a wrong offset, a state gradient filed under another sequence, or a dropped
    sum over sequences fails here. Includes an empty sequence and unused tokens."""
    rng = np.random.default_rng(11)
    H, lengths, dk, dv = 2, [3, 0, 4], 4, 3
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, lengths, dk, dv, gap=2)
    N = len(lengths)
    x = dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=Ip,
             mu0=rng.standard_normal((N, H, dv, dk)), I0=rng.uniform(0.5, 2.0, (N, H, dv, dk)))
    dy = rng.standard_normal(v.shape)
    dmu = rng.standard_normal((N, H, dv, dk))
    dI = rng.standard_normal((N, H, dv, dk))
    g = ovl.gradients(x, cu, dy, dmu, dI)
    eps = 1e-6
    for name in ("q", "k", "v", "beta", "d_t", "A", "I_prior", "mu0", "I0"):
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            keep = x[name][idx]
            x[name][idx] = keep + eps
            lp = _packed_loss(x, cu, dy, dmu, dI)
            x[name][idx] = keep - eps
            lm = _packed_loss(x, cu, dy, dmu, dI)
            x[name][idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_packed_gradients_of_empty_sequences_and_unused_tokens():
    """An empty sequence hands its state through unchanged, so its initial-state
    gradients are the final-state ones exactly; tokens outside every sequence
    get zero gradients."""
    rng = np.random.default_rng(12)
    H, lengths, dk, dv = 2, [0, 5, 0], 4, 3
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, lengths, dk, dv, gap=3)
    N = len(lengths)
    x = dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=Ip,
             mu0=rng.standard_normal((N, H, dv, dk)), I0=rng.uniform(0.5, 2.0, (N, H, dv, dk)))
    dmu = rng.standard_normal((N, H, dv, dk))
    dI = rng.standard_normal((N, H, dv, dk))
    g = ovl.gradients(x, cu, rng.standard_normal(v.shape), dmu, dI)
    for n in (0, 2):
        np.testing.assert_array_equal(g["mu0"][n], dmu[n])
        np.testing.assert_array_equal(g["I0"][n], dI[n])
    for name in ("q", "k", "v", "beta", "d_t"):
        assert not g[name][:, 5:].any(), name


def test_packed_gradients_when_the_loss_reaches_no_input():
    """Empty sequences with no final-state cotangent: the loss does not depend on
    their inputs, so their gradients are zero (with and without an initial state),
    and A and I_prior get exactly the non-empty sequence's own gradients."""
    from oracle import autograd as ag
    rng = np.random.default_rng(13)
    H, lengths, dk, dv = 2, [0, 4, 0], 4, 3
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, lengths, dk, dv)
    N = len(lengths)
    for with_state in (False, True):
        x = dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=Ip,
                 mu0=rng.standard_normal((N, H, dv, dk)) if with_state else None,
                 I0=rng.uniform(0.5, 2.0, (N, H, dv, dk)) if with_state else None)
        dy = rng.standard_normal(v.shape)
        g = ovl.gradients(x, cu, dy)
        one = {n: x[n][None] for n in ("q", "k", "v", "beta", "d_t")}
        one.update(A=A, I_prior=Ip, mu0=None if x["mu0"] is None else x["mu0"][1:2],
                   I0=None if x["I0"] is None else x["I0"][1:2])
        g1 = ag.gradients(one, dy[None])
        for name in ("A", "I_prior"):
            np.testing.assert_array_equal(g[name], g1[name], err_msg=name)
        if with_state:
            for n in (0, 2):
                assert not g["mu0"][n].any() and not g["I0"][n].any()
    # a single empty sequence with no cotangent at all
    q, k, v, beta, d_t, A, Ip, cu = _packed(rng, H, [0], dk, dv)
    g = ovl.gradients(dict(q=q, k=k, v=v, beta=beta, d_t=d_t, A=A, I_prior=Ip), cu, np.zeros(v.shape))
    assert not g["A"].any() and not g["I_prior"].any()
