"""GPU parity of the fused prologue (palimpsa_forward_fused, palimpsa_step_fused)
against the fp64 oracle's prologue + recurrence on the same raw inputs.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 10 (q/k L2 norm of Palimpsa-D), slide 11 (v*
input, per-head b_scale); the activations are the workload recipes'."""
import numpy as np
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import synthetic as syn
from metaplastic_linear_attention_gb300.synthetic import as_float64_numpy as f64
from oracle import prologue as opro
from tests._helpers import TIGHT, pick, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"

FLAG_SETS = [dict(qk_norm=False, v_star=False), dict(qk_norm=True, v_star=False),
             dict(qk_norm=False, v_star=True), dict(qk_norm=True, v_star=True)]


def _raw(B, H, T, dk, dv, bf16, seed, b_scale=True):
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16, seed=seed)
    inp = syn.sequence_inputs(wl, raw=True)
    if not b_scale:
        inp["b_scale"] = None
    return inp


def _oracle(inp, mu0=None, I0=None, **flags):
    bs = None if inp["b_scale"] is None else f64(inp["b_scale"])
    return opro.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["beta_raw"]), f64(inp["d_raw"]),
                        f64(inp["A"]), f64(inp["I_prior"]), b_scale=bs,
                        mu0=None if mu0 is None else f64(mu0), I0=None if I0 is None else f64(I0), **flags)


def _gpu_fused(inp, mu0=None, I0=None, chunk=0, **flags):
    g = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    out = pal.palimpsa_forward_fused(g["q"], g["k"], g["v"], g["beta_raw"], g["d_raw"], g["A"], g["I_prior"],
                                     g["b_scale"], None if mu0 is None else mu0.to(DEV),
                                     None if I0 is None else I0.to(DEV), chunk=chunk, **flags)
    assert pal.palimpsa_get_device_status() == 0
    return out


def _check(out, ref):
    errs = [rel_l2(o.cpu().numpy() if torch.is_tensor(o) else o, r) for o, r in zip(out, ref)]
    assert max(errs) <= TIGHT, errs
    return errs


CASES = [
    # (B, H, T, d_k, d_v, bf16, chunk, segments)
    (1, 2, 1, 128, 64, True, 16, 1),
    (2, 3, 77, 128, 64, True, 32, 1),
    (1, 2, 130, 64, 40, False, 16, 1),
    (2, 2, 200, 128, 64, True, 32, 3),   # time split: pass A applies the prologue too
    (1, 3, 161, 64, 64, False, 16, 4),
    (1, 1, 97, 128, 256, False, 32, 2),
]


@pytest.mark.parametrize("flags", FLAG_SETS, ids=["plain", "qknorm", "vstar", "qknorm_vstar"])
@pytest.mark.parametrize("B,H,T,dk,dv,bf16,chunk,S", CASES)
def test_fused_forward_matches_oracle(B, H, T, dk, dv, bf16, chunk, S, flags):
    inp = _raw(B, H, T, dk, dv, bf16, seed=1000 + T + dk + dv)
    ref = _oracle(inp, **flags)
    pal.palimpsa_set_forward_segments(S)
    try:
        out = _gpu_fused(inp, chunk=chunk, **flags)
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check(out, ref)


@pytest.mark.parametrize("S", [1, 3])
def test_fused_forward_initial_state_and_no_b_scale(S):
    inp = _raw(2, 2, 150, 128, 64, True, seed=77, b_scale=False)
    g = torch.Generator().manual_seed(5)
    mu0 = torch.randn((2, 2, 64, 128), generator=g)
    I0 = 0.5 + 3.0 * torch.rand((2, 2, 64, 128), generator=g)
    ref = _oracle(inp, mu0, I0, qk_norm=True, v_star=True)
    pal.palimpsa_set_forward_segments(S)
    try:
        out = _gpu_fused(inp, mu0, I0, qk_norm=True, v_star=True)
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check(out, ref)


@pytest.mark.parametrize("name,heads,flags", [
    ("small_layer", [(0, 0), (1, 7), (3, 15)], dict(qk_norm=True, v_star=False)),
    ("layer_760m", [(0, 0), (5, 11), (7, 23)], dict(qk_norm=True, v_star=True)),
])
def test_fused_full_size_sampled_heads(name, heads, flags):
    """The whole workload on the GPU in the launch configuration the library picks;
    the oracle on sampled heads (heads are independent)."""
    wl = syn.WORKLOADS[name]
    inp = syn.sequence_inputs(wl, raw=True)
    out = _gpu_fused(inp, chunk=wl.chunk, **flags)
    hs = [h for _, h in heads]
    bs = f64(inp["b_scale"])[hs]
    ref = opro.forward(pick(inp["q"], heads), pick(inp["k"], heads), pick(inp["v"], heads),
                       pick(inp["beta_raw"], heads), pick(inp["d_raw"], heads), f64(inp["A"])[hs],
                       f64(inp["I_prior"])[hs], b_scale=bs, **flags)
    _check([pick(o, heads) for o in out], ref)


STEP_CASES = [(4, 3, 128, 64, True), (3, 2, 64, 40, False), (2, 2, 128, 256, False)]


@pytest.mark.parametrize("flags", FLAG_SETS, ids=["plain", "qknorm", "vstar", "qknorm_vstar"])
@pytest.mark.parametrize("B,H,dk,dv,bf16", STEP_CASES)
def test_fused_step_matches_oracle(B, H, dk, dv, bf16, flags):
    wl = syn.WORKLOADS["decode"].with_(B=B, H=H, d_k=dk, d_v=dv, bf16=bf16, seed=B * 100 + dk + dv)
    pre = syn.sequence_inputs(wl, T=1, raw=True)
    steps = syn.decode_inputs(wl, 6, raw=True)
    g = torch.Generator().manual_seed(B + H)
    mu = torch.randn((B, H, dv, dk), generator=g)
    I = 0.5 + 2.0 * torch.rand((B, H, dv, dk), generator=g)
    mu_ref, I_ref = f64(mu), f64(I)
    mu_d, I_d = mu.to(DEV), I.to(DEV)
    A, Ip, bsc = pre["A"].to(DEV), pre["I_prior"].to(DEV), pre["b_scale"].to(DEV)
    for t in range(6):
        y = pal.palimpsa_step_fused(steps["q"][t].to(DEV), steps["k"][t].to(DEV), steps["v"][t].to(DEV),
                                    steps["beta_raw"][t].to(DEV), steps["d_raw"][t].to(DEV), A, Ip, mu_d, I_d,
                                    bsc, **flags)
        y_ref, mu_ref, I_ref = opro.step(f64(steps["q"][t]), f64(steps["k"][t]), f64(steps["v"][t]),
                                         f64(steps["beta_raw"][t]), f64(steps["d_raw"][t]), f64(pre["A"]),
                                         f64(pre["I_prior"]), mu_ref, I_ref, b_scale=f64(pre["b_scale"]), **flags)
        assert rel_l2(y.cpu().numpy(), y_ref) <= TIGHT
    assert pal.palimpsa_get_device_status() == 0
    assert rel_l2(mu_d.cpu().numpy(), mu_ref) <= TIGHT
    assert rel_l2(I_d.cpu().numpy(), I_ref) <= TIGHT


def test_fused_step_equals_one_token_fused_forward():
    wl = syn.WORKLOADS["small_layer"].with_(B=3, H=2, seed=4242)
    inp = syn.sequence_inputs(wl, T=1, raw=True)
    g = {k: v.to(DEV) for k, v in inp.items()}
    y, muT, IT = pal.palimpsa_forward_fused(g["q"], g["k"], g["v"], g["beta_raw"], g["d_raw"], g["A"], g["I_prior"],
                                            g["b_scale"], qk_norm=True, v_star=True)
    mu = torch.zeros_like(muT)
    I = g["I_prior"][None, :, None, None].expand_as(IT).contiguous()
    ys = pal.palimpsa_step_fused(g["q"][:, :, 0], g["k"][:, :, 0], g["v"][:, :, 0], g["beta_raw"][:, :, 0],
                                 g["d_raw"][:, :, 0], g["A"], g["I_prior"], mu, I, g["b_scale"], qk_norm=True,
                                 v_star=True)
    assert rel_l2(ys.cpu().numpy(), y[:, :, 0].cpu().numpy()) < 1e-6
    assert rel_l2(mu.cpu().numpy(), muT.cpu().numpy()) < 1e-6
    assert rel_l2(I.cpu().numpy(), IT.cpu().numpy()) < 1e-6


def test_negative_b_scale_is_reported_not_faulted():
    inp = _raw(1, 2, 40, 128, 64, True, seed=9)
    g = {k: v.to(DEV) for k, v in inp.items()}
    bad = g["b_scale"].clone()
    bad[1] = -0.5
    pal.palimpsa_forward_fused(g["q"], g["k"], g["v"], g["beta_raw"], g["d_raw"], g["A"], g["I_prior"], bad)
    assert pal.palimpsa_get_device_status() == 5  # PALIMPSA_ERR_DOMAIN
    # the context stays usable
    out = _gpu_fused(inp, qk_norm=True)
    _check(out, _oracle(inp, qk_norm=True))


@pytest.mark.parametrize("flags", FLAG_SETS, ids=["plain", "qknorm", "vstar", "qknorm_vstar"])
def test_fused_step_sequence_equals_token_by_token_bitwise(flags):
    """One palimpsa_step_sequence_fused call (4-D raw inputs) enqueues the same
    launches as S palimpsa_step_fused calls: identical bits."""
    wl = syn.WORKLOADS["decode"].with_(B=3, H=2, seed=515)
    pre = syn.sequence_inputs(wl, T=1, raw=True)
    steps = {n: t.to(DEV) for n, t in syn.decode_inputs(wl, 7, raw=True).items()}
    A, Ip, bsc = pre["A"].to(DEV), pre["I_prior"].to(DEV), pre["b_scale"].to(DEV)
    g = torch.Generator().manual_seed(516)
    mu0 = torch.randn((3, 2, 64, 128), generator=g).to(DEV)
    I0 = (0.5 + torch.rand((3, 2, 64, 128), generator=g)).to(DEV)
    mu_a, I_a = mu0.clone(), I0.clone()
    y_a = pal.palimpsa_step_fused(steps["q"], steps["k"], steps["v"], steps["beta_raw"], steps["d_raw"], A, Ip, mu_a,
                                  I_a, bsc, **flags)
    mu_b, I_b = mu0.clone(), I0.clone()
    y_b = torch.stack([pal.palimpsa_step_fused(steps["q"][t], steps["k"][t], steps["v"][t], steps["beta_raw"][t],
                                               steps["d_raw"][t], A, Ip, mu_b, I_b, bsc, **flags) for t in range(7)])
    assert pal.palimpsa_get_device_status() == 0
    assert torch.equal(y_a, y_b) and torch.equal(mu_a, mu_b) and torch.equal(I_a, I_b)
