"""Randomised GPU parity: seeded draws of shapes, dtypes, staging chunks, forced
segment counts (the time split), initial states and gate statistics, each run
through the chunked forward, a few decode steps and the backward, and checked
against the fp64 oracle (forward and steps) and fp64 autograd on the oracle's
recurrence (backward) at 1e-4 relative L2 per output. dA, a per-head sum over
every token whose terms can cancel by three orders of magnitude (or exactly), is
checked through its linear relation to dd_t (tests/_helpers.py, dA_within_bar).

The draws cover the corners the hand-written cases visit one at a time:
d_k in {64, 128}; d_v from 8 to 256 (multiples of 8, which select every CTA row
grouping and, at d_k = 128 with d_v a multiple of 32 and bf16 inputs, the
tensor-core pass A); T from 1 to a few hundred tokens, ragged against the
32-token chunk and checkpoint spacing; 1 to 9 segments; long and short memory;
the backward with recomputed states or with the checkpointed forward's. Packed
batches draw 1 to 6 sequence lengths (empty ones among them) the same way and run
the packed forward and the packed training pair against the oracle run per
sequence.
"""
import numpy as np
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
import oracle
from metaplastic_linear_attention_gb300 import synthetic as syn
from oracle import varlen as ovl
from tests._helpers import TIGHT, dA_within_bar, oracle_forward_from, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_CASES = 48
N_PACKED = 24


def _draw_case(i):
    r = np.random.default_rng(9000 + i)
    dk = int(r.choice([64, 128]))
    dv = int(r.choice([8, 16, 24, 32, 40, 64, 96, 128, 256]))
    return dict(
        B=int(r.integers(1, 4)), H=int(r.integers(1, 4)), T=int(r.choice([1, 7, 31, 32, 33, 97, 160, 257, 300])),
        d_k=dk, d_v=dv, bf16=bool(r.integers(0, 2)), chunk=int(r.choice([0, 16, 32, 64, 128])),
        segments=int(r.choice([0, 1, 2, 3, 5, 9])), dt_mean=float(r.choice([-2.0, -1.0, 0.0, 1.0])),
        with_state=bool(r.integers(0, 2)), seed=int(r.integers(1, 1 << 30)), ckpt=bool(r.integers(0, 2)))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_forward_steps_backward(i):
    c = _draw_case(i)
    wl = syn.WORKLOADS["small_layer"].with_(B=c["B"], H=c["H"], T=c["T"], d_k=c["d_k"], d_v=c["d_v"],
                                            bf16=c["bf16"], chunk=c["chunk"], dt_mean=c["dt_mean"])
    inp = syn.sequence_inputs(wl, seed=c["seed"])
    g = torch.Generator().manual_seed(c["seed"] + 1)
    shape = (c["B"], c["H"], c["d_v"], c["d_k"])
    mu0 = torch.randn(shape, generator=g) if c["with_state"] else None
    I0 = (0.5 + 3.0 * torch.rand(shape, generator=g)) if c["with_state"] else None
    gi = {k: v.to(DEV) for k, v in inp.items()}
    d = lambda t: None if t is None else t.to(DEV)

    # forward, with the drawn segment count forced (0: the planner's choice)
    pal.palimpsa_set_forward_segments(c["segments"])
    try:
        y, mu, I = pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                                gi["I_prior"], d(mu0), d(I0), chunk=c["chunk"])
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0, c
    ry, rmu, rI = oracle_forward_from(inp, mu0, I0)
    for name, got, ref in (("y", y, ry), ("mu_T", mu, rmu), ("I_T", I, rI)):
        assert rel_l2(got.cpu().numpy(), ref) <= TIGHT, (name, c)

    # three decode steps from the final state
    steps = syn.decode_inputs(wl, 3, seed=c["seed"] + 2)
    f = syn.as_float64_numpy
    for s in range(3):
        gs = {k: v[s].to(DEV) for k, v in steps.items()}
        ys = pal.palimpsa_step(gs["q"], gs["k"], gs["v"], gs["beta"], gs["d_t"], gi["A"], gi["I_prior"], mu, I)
        rys, rmu, rI = oracle.step(*(f(steps[n][s]) for n in ("q", "k", "v", "beta", "d_t")), f(inp["A"]),
                                   f(inp["I_prior"]), rmu, rI)
        assert rel_l2(ys.cpu().numpy(), rys) <= TIGHT, ("step", s, c)
    assert pal.palimpsa_get_device_status() == 0, c
    assert rel_l2(mu.cpu().numpy(), rmu) <= TIGHT and rel_l2(I.cpu().numpy(), rI) <= TIGHT, c

    # backward of <dy, y> (and of the final state) against fp64 autograd
    from oracle import autograd as ag
    dy = torch.randn((c["B"], c["H"], c["T"], c["d_v"]), generator=g)
    dmu = torch.randn(shape, generator=g)
    dI = torch.randn(shape, generator=g)
    ref = ag.gradients({n: (None if t is None else f(t)) for n, t in
                        dict(q=inp["q"], k=inp["k"], v=inp["v"], beta=inp["beta"], d_t=inp["d_t"], A=inp["A"],
                             I_prior=inp["I_prior"], mu0=mu0, I0=I0).items()}, f(dy), f(dmu), f(dI))
    ck = None
    if c["ckpt"]:
        *_, ck = pal.palimpsa_forward_checkpointed(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                                   gi["I_prior"], d(mu0), d(I0), chunk=c["chunk"])
    out = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], d(mu0),
                                d(I0), d(dy), d(dmu), d(dI), ckpt=ck)
    assert pal.palimpsa_get_device_status() == 0, c
    pairs = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t"),
             ("dI_prior", "I_prior"), ("dmu0", "mu0"), ("dI0", "I0")]
    for n, m in pairs:
        if c["with_state"] or n not in ("dmu0", "dI0"):
            assert rel_l2(out[n].cpu(), ref[m]) <= TIGHT, (n, c)
    ok, detail = dA_within_bar(out["dA"].cpu(), ref["A"], out["dd_t"].cpu(), ref["d_t"], f(inp["d_t"]),
                               f(inp["A"]))
    assert ok, ("dA", detail, c)


def _draw_packed(i):
    r = np.random.default_rng(9500 + i)
    n = int(r.integers(1, 7))
    return dict(lengths=[int(x) for x in r.choice([0, 1, 5, 31, 32, 33, 64, 97, 160, 300], size=n)],
                H=int(r.integers(1, 4)), d_k=int(r.choice([64, 128])),
                d_v=int(r.choice([8, 16, 24, 32, 40, 64, 96, 128, 256])), bf16=bool(r.integers(0, 2)),
                chunk=int(r.choice([0, 16, 32, 64, 128])), segments=int(r.choice([0, 0, 2, 3, 5])),
                dt_mean=float(r.choice([-2.0, -1.0, 0.0, 1.0])), with_state=bool(r.integers(0, 2)),
                with_final=bool(r.integers(0, 2)), ckpt=bool(r.integers(0, 2)), seed=int(r.integers(1, 1 << 30)))


@pytest.mark.parametrize("i", range(N_PACKED))
def test_random_packed_batch_forward_and_training_pair(i):
    c = _draw_packed(i)
    wl = syn.WORKLOADS["small_layer"].with_(d_k=c["d_k"], d_v=c["d_v"], bf16=c["bf16"], dt_mean=c["dt_mean"],
                                            seed=c["seed"])
    inp = syn.packed_inputs(wl, c["lengths"], H=c["H"])
    N, H, total = len(c["lengths"]), c["H"], inp["q"].shape[1]
    g = torch.Generator().manual_seed(c["seed"] + 1)
    shape = (N, H, c["d_v"], c["d_k"])
    mu0 = torch.randn(shape, generator=g) if c["with_state"] else None
    I0 = (0.5 + 3.0 * torch.rand(shape, generator=g)) if c["with_state"] else None
    dy = torch.randn((H, total, c["d_v"]), generator=g)
    dmu = torch.randn(shape, generator=g) if c["with_final"] else None
    dI = torch.randn(shape, generator=g) if c["with_final"] else None
    f = syn.as_float64_numpy
    fo = lambda t: None if t is None else f(t)
    d = lambda t: None if t is None else t.to(DEV)
    gi = {k: v.to(DEV) for k, v in inp.items()}
    cu = inp["cu_seqlens"].tolist()
    x = {n: f(inp[n]) for n in ("q", "k", "v", "beta", "d_t", "A", "I_prior")}

    pal.palimpsa_set_forward_segments(c["segments"])
    try:
        out = pal.palimpsa_forward_varlen(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"],
                                          gi["cu_seqlens"], d(mu0), d(I0), chunk=c["chunk"])
        ck = None
        if c["ckpt"]:
            *_, ck = pal.palimpsa_forward_varlen_checkpointed(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"],
                                                              gi["A"], gi["I_prior"], gi["cu_seqlens"], d(mu0),
                                                              d(I0), chunk=c["chunk"])
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0, c
    ref = ovl.forward(*x.values(), cu, mu0=fo(mu0), I0=fo(I0))
    for name, got, want in zip(("y", "mu_T", "I_T"), out, ref):
        assert rel_l2(got.cpu().numpy(), want) <= TIGHT, (name, c)

    grads = pal.palimpsa_backward_varlen(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"],
                                         gi["cu_seqlens"], d(mu0), d(I0), d(dy), d(dmu), d(dI), ckpt=ck)
    assert pal.palimpsa_get_device_status() == 0, c
    rg = ovl.gradients(dict(x, mu0=fo(mu0), I0=fo(I0)), cu, f(dy), fo(dmu), fo(dI))
    pairs = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t"),
             ("dI_prior", "I_prior")] + ([("dmu0", "mu0"), ("dI0", "I0")] if c["with_state"] else [])
    for n, m in pairs:
        assert rel_l2(grads[n].cpu().numpy(), rg[m]) <= TIGHT, (n, c)
    ok, detail = dA_within_bar(grads["dA"].cpu(), rg["A"], grads["dd_t"].cpu(), rg["d_t"], x["d_t"], x["A"])
    assert ok, ("dA", detail, c)


# ------------------------------------------------------------ the tensor-core summaries
N_TC = 24


def _draw_tc(i):
    """A time split whose summaries run on the tensor cores (bf16 inputs, d_k = 128,
    d_v a multiple of 32 up to 128), with ragged segment ends and, for half the
    draws, the fused prologue (its q/k norm and v* modes reach the summaries too)."""
    r = np.random.default_rng(9800 + i)
    fused = bool(r.integers(0, 2))
    return dict(B=int(r.integers(1, 3)), H=int(r.integers(1, 4)), T=int(r.choice([33, 65, 100, 257, 511, 700])),
                d_v=int(r.choice([32, 64, 96, 128])), segments=int(r.integers(2, 10)),
                dt_mean=float(r.choice([-2.0, -1.0, 0.0])), with_state=bool(r.integers(0, 2)), fused=fused,
                qk_norm=fused and bool(r.integers(0, 2)), v_star=fused and bool(r.integers(0, 2)),
                seed=int(r.integers(1, 1 << 30)))


@pytest.mark.parametrize("i", range(N_TC))
def test_random_time_split_on_the_tensor_cores(i):
    from oracle import prologue as opro
    c = _draw_tc(i)
    wl = syn.WORKLOADS["small_layer"].with_(B=c["B"], H=c["H"], T=c["T"], d_k=128, d_v=c["d_v"], bf16=True,
                                            dt_mean=c["dt_mean"], seed=c["seed"])
    plan = pal.palimpsa_forward_plan(c["B"], c["H"], c["T"], 128, c["d_v"], bf16=True)
    g = torch.Generator().manual_seed(c["seed"] + 1)
    shape = (c["B"], c["H"], c["d_v"], 128)
    mu0 = torch.randn(shape, generator=g) if c["with_state"] else None
    I0 = (0.5 + 3.0 * torch.rand(shape, generator=g)) if c["with_state"] else None
    d = lambda t: None if t is None else t.to(DEV)
    f = syn.as_float64_numpy
    fo = lambda t: None if t is None else f(t)
    pal.palimpsa_set_forward_segments(c["segments"])
    try:
        seg = pal.palimpsa_forward_plan(c["B"], c["H"], c["T"], 128, c["d_v"], bf16=True)["segments"]
        if c["fused"]:
            inp = syn.sequence_inputs(wl, raw=True)
            gi = {k: d(v) for k, v in inp.items()}
            out = pal.palimpsa_forward_fused(gi["q"], gi["k"], gi["v"], gi["beta_raw"], gi["d_raw"], gi["A"],
                                             gi["I_prior"], gi["b_scale"], d(mu0), d(I0), qk_norm=c["qk_norm"],
                                             v_star=c["v_star"])
            ref = opro.forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["beta_raw"]), f(inp["d_raw"]),
                               f(inp["A"]), f(inp["I_prior"]), b_scale=f(inp["b_scale"]), mu0=fo(mu0), I0=fo(I0),
                               qk_norm=c["qk_norm"], v_star=c["v_star"])
        else:
            inp = syn.sequence_inputs(wl)
            gi = {k: d(v) for k, v in inp.items()}
            out = pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                               gi["I_prior"], d(mu0), d(I0))
            ref = oracle_forward_from(inp, mu0, I0)
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert seg > 1, (c, plan)
    assert pal.palimpsa_get_device_status() == 0, c
    for name, got, want in zip(("y", "mu_T", "I_T"), out, ref):
        assert rel_l2(got.cpu().numpy(), want) <= TIGHT, (name, c)
