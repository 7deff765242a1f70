"""GPU parity of the time-sharded forward's kernels: palimpsa_segment_summary and
palimpsa_state_combine against the fp64 oracle, and R time shards run one after
another in one process (the exchange reduced to stacking the summaries, which
the gloo test of ``tsplit`` covers across processes) against one oracle pass.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 9 (App. A.12): the natural-parameter
recurrences are affine in the state with the shared decay alpha."""
import numpy as np
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import synthetic as syn
from metaplastic_linear_attention_gb300.synthetic import as_float64_numpy as f64
from tests._helpers import TIGHT, oracle_forward_from, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu(d):
    return {k: v.to(DEV) for k, v in d.items()}


def _sl(inp, t0, t1):
    out = dict(inp)
    for name in ("q", "k", "v", "beta", "d_t"):
        out[name] = inp[name][:, :, t0:t1].contiguous()
    return out


@pytest.mark.parametrize("B,H,T,dk,dv,bf16,S", [
    (2, 2, 1, 128, 64, True, 0), (1, 3, 77, 64, 40, False, 0), (2, 2, 400, 128, 64, True, 4),
    (1, 2, 1000, 128, 64, False, 0), (1, 1, 0, 128, 64, True, 0),
])
def test_segment_summary_is_the_state_from_zero(B, H, T, dk, dv, bf16, S):
    """From a zero excess state the summary is the final state itself: dM = mu_T I_T,
    dIbar = I_T - I_prior; Gamma = exp(-A sum_t d_t) (the product of the alphas)."""
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16, seed=T + dk)
    inp = syn.sequence_inputs(wl)
    pal.palimpsa_set_forward_segments(S)
    try:
        g = _gpu(inp)
        summ, gam = pal.palimpsa_segment_summary(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"],
                                                 g["I_prior"])
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0
    Ip = f64(inp["I_prior"])[None, :, None, None]
    gamma_ref = np.exp(-f64(inp["A"])[None, :] * f64(inp["d_t"]).sum(-1))
    np.testing.assert_allclose(gam.cpu().numpy(), gamma_ref, rtol=1e-4, atol=1e-30)
    if T == 0:
        assert torch.count_nonzero(summ) == 0
        return
    _, mu, I = oracle_forward_from(inp)
    assert rel_l2(summ[:, :, 0].cpu().numpy(), mu * I) <= TIGHT
    assert rel_l2(summ[:, :, 1].cpu().numpy(), I - Ip) <= TIGHT


@pytest.mark.parametrize("bounds,bf16,with_state", [
    ([0, 100, 300], True, False), ([0, 1, 129, 129, 500], False, True), ([0, 700, 1500, 3000], True, True),
])
def test_time_shards_in_sequence_equal_one_pass(bounds, bf16, with_state):
    B, H, dk, dv = 1, 2, 128, 64
    T = bounds[-1]
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, bf16=bf16, seed=len(bounds) + T)
    inp = syn.sequence_inputs(wl)
    mu0 = I0 = None
    if with_state:
        gg = torch.Generator().manual_seed(2)
        mu0 = torch.randn((B, H, dv, dk), generator=gg)
        I0 = 0.5 + 3.0 * torch.rand((B, H, dv, dk), generator=gg)
    y_ref, mu_ref, I_ref = oracle_forward_from(inp, mu0=mu0, I0=I0)
    g = _gpu(inp)
    m0 = None if mu0 is None else mu0.to(DEV)
    i0 = None if I0 is None else I0.to(DEV)
    R = len(bounds) - 1
    shards = [_sl(g, bounds[r], bounds[r + 1]) for r in range(R)]
    # step 1 on every "rank", then the exchange (stacking), then steps 3-4 per rank
    summ = [pal.palimpsa_segment_summary(s["q"], s["k"], s["v"], s["beta"], s["d_t"], g["A"], g["I_prior"])
            for s in shards]
    S_all = torch.stack([s for s, _ in summ])
    G_all = torch.stack([gm for _, gm in summ])
    for r, s in enumerate(shards):
        mu_s, I_s = pal.palimpsa_state_combine(S_all[:r], G_all[:r], g["I_prior"], m0, i0)
        y, mu, I = pal.palimpsa_forward_chunked(s["q"], s["k"], s["v"], s["beta"], s["d_t"], g["A"], g["I_prior"],
                                                mu_s, I_s)
        assert pal.palimpsa_get_device_status() == 0
        if bounds[r + 1] > bounds[r]:
            assert rel_l2(y.cpu().numpy(), y_ref[:, :, bounds[r]:bounds[r + 1]]) <= TIGHT
    assert rel_l2(mu.cpu().numpy(), mu_ref) <= TIGHT
    assert rel_l2(I.cpu().numpy(), I_ref) <= TIGHT


def test_state_combine_of_nothing_is_the_initial_state_in_place():
    B, H, dv, dk = 2, 3, 64, 128
    gg = torch.Generator().manual_seed(4)
    mu0 = torch.randn((B, H, dv, dk), generator=gg).to(DEV)
    I0 = (0.5 + torch.rand((B, H, dv, dk), generator=gg)).to(DEV)
    Ip = torch.ones(H, device=DEV)
    mu_keep, I_keep = mu0.clone(), I0.clone()
    S = torch.empty((0, B, H, 2, dv, dk), device=DEV)
    G = torch.empty((0, B, H), device=DEV)
    mu, I = pal.palimpsa_state_combine(S, G, Ip, mu0, I0, mu_out=mu0, I_out=I0)
    assert torch.equal(I, I_keep)
    assert rel_l2(mu.cpu().numpy(), mu_keep.cpu().numpy()) < 2e-7   # (I0 mu0) / I0
    mu_d, I_d = pal.palimpsa_state_combine(S, G, Ip)
    assert torch.count_nonzero(mu_d) == 0 and torch.equal(I_d, torch.ones_like(I_d))


def test_state_combine_domain_violation_is_reported_not_faulted():
    """palimpsa_state_combine reports a non-positive I_prior or I0 without a fault."""
    g = torch.Generator().manual_seed(5)
    summ = torch.rand((1, 1, 2, 2, 64, 128), generator=g).to(DEV)   # R = 1, B = 1, H = 2
    gam = torch.rand((1, 1, 2), generator=g).to(DEV)
    I_prior = torch.ones(2, device=DEV)
    mu0 = torch.zeros((1, 2, 64, 128), device=DEV)
    I0 = torch.ones((1, 2, 64, 128), device=DEV)
    bad_I0 = I0.clone()
    bad_I0[0, 1, 5, 6] = -1.0
    pal.palimpsa_state_combine(summ, gam, I_prior, mu0, bad_I0)
    assert pal.palimpsa_get_device_status() == 5          # PALIMPSA_ERR_DOMAIN
    pal.palimpsa_state_combine(summ, gam, torch.tensor([1.0, 0.0], device=DEV), mu0, I0)
    assert pal.palimpsa_get_device_status() == 5
    pal.palimpsa_state_combine(summ, gam, I_prior, mu0, I0)
    assert pal.palimpsa_get_device_status() == 0
