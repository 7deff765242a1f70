"""Agreement between the oracle's independent statements of the recurrence:
the C token-by-token scan, the NumPy mean/precision form and the NumPy chunked
natural-parameter form (slide 9 / App. A.12 of the Palimpsa slide deck: the
natural parameters turn Eq. (5) into two affine scans, evaluated in parallel
inside a chunk and carried sequentially between chunks)."""
import numpy as np
import pytest

import oracle
from oracle import reference_np as rnp


def _problem(seed, B, H, T, dk, dv, prior_full=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, H, T, dv))))
    d_t = np.log1p(np.exp(rng.standard_normal((B, H, T))))
    A = np.full(H, 0.5) if H == 2 else rng.uniform(0.1, 1.0, H)
    I_prior = rng.uniform(0.5, 2.0, (H, dv, dk)) if prior_full else np.ones(H)
    return q, k, v, beta, d_t, A, I_prior


def test_c_matches_numpy_at_tiny_config_shape():
    """B=1, H=2, T=256, d_k=d_v=64 (the fp32 tiny-sequence shape): the two
    separately written fp64 statements agree to round-off."""
    args = _problem(0, 1, 2, 256, 64, 64)
    y, muT, IT = oracle.forward(*args)
    yn, mun, In = rnp.forward_mu_form(*args)
    for a, b in ((y, yn), (muT, mun), (IT, In)):
        assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-13


def test_c_matches_numpy_with_initial_state_and_per_state_prior():
    q, k, v, beta, d_t, A, I_prior = _problem(1, 2, 3, 40, 8, 5, prior_full=True)
    rng = np.random.default_rng(2)
    mu0 = rng.standard_normal((2, 3, 5, 8))
    I0 = rng.uniform(0.3, 4.0, (2, 3, 5, 8))
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    yn, mun, In = rnp.forward_mu_form(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    np.testing.assert_allclose(y, yn, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(muT, mun, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(IT, In, rtol=1e-13)


@pytest.mark.parametrize("chunk", [1, 7, 16, 64, 100])
def test_chunked_natural_form_equals_sequential(chunk):
    q, k, v, beta, d_t, A, I_prior = _problem(3, 1, 2, 100, 6, 4)
    rng = np.random.default_rng(4)
    mu0 = rng.standard_normal((1, 2, 4, 6))
    I0 = rng.uniform(0.5, 3.0, (1, 2, 4, 6))
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    yc, muc, Ic = rnp.forward_natural_chunked(q, k, v, beta, d_t, A, I_prior, chunk, mu0=mu0, I0=I0)
    for a, b in ((yc, y), (muc, muT), (Ic, IT)):
        assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-12


def test_step_equals_one_token_forward_and_continuation():
    """Decoding token by token with the step equals the T-token scan, and a scan
    split at any point and resumed from its (mu_T, I_T) equals the whole scan."""
    q, k, v, beta, d_t, A, I_prior = _problem(5, 2, 2, 30, 8, 4)
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior)
    mu = np.zeros_like(muT)
    I = np.broadcast_to(I_prior[None, :, None, None], muT.shape).copy()
    for t in range(30):
        yt, mu, I = oracle.step(q[:, :, t], k[:, :, t], v[:, :, t], beta[:, :, t], d_t[:, :, t], A,
                                I_prior, mu, I)
        np.testing.assert_array_equal(yt, y[:, :, t])
    np.testing.assert_array_equal(mu, muT)
    np.testing.assert_array_equal(I, IT)
    s = 13
    y1, m1, i1 = oracle.forward(q[:, :, :s], k[:, :, :s], v[:, :, :s], beta[:, :, :s], d_t[:, :, :s], A, I_prior)
    y2, m2, i2 = oracle.forward(q[:, :, s:], k[:, :, s:], v[:, :, s:], beta[:, :, s:], d_t[:, :, s:], A, I_prior,
                                mu0=m1, I0=i1)
    np.testing.assert_array_equal(np.concatenate([y1, y2], axis=2), y)
    np.testing.assert_array_equal(m2, muT)
    np.testing.assert_array_equal(i2, IT)


def test_thread_count_does_not_change_results():
    args = _problem(6, 2, 2, 50, 16, 8)
    a = oracle.forward(*args, nthreads=1)
    b = oracle.forward(*args, nthreads=4)
    for x, z in zip(a, b):
        np.testing.assert_array_equal(x, z)


def test_empty_sequence_returns_initial_state():
    q, k, v, beta, d_t, A, I_prior = _problem(7, 1, 2, 0, 4, 3)
    rng = np.random.default_rng(8)
    mu0 = rng.standard_normal((1, 2, 3, 4))
    I0 = rng.uniform(0.5, 2, (1, 2, 3, 4))
    y, muT, IT = oracle.forward(q, k, v, beta, d_t, A, I_prior, mu0=mu0, I0=I0)
    assert y.shape == (1, 2, 0, 3)
    np.testing.assert_array_equal(muT, mu0)
    np.testing.assert_array_equal(IT, I0)
