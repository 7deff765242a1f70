"""GPU parity: the CUDA kernels, called through the C ABI, against the fp64
oracle on the same seeded inputs (relative L2 per output tensor).

Small cases run the oracle on everything; the full-size workloads run the GPU
on the whole problem in the launch configuration the benchmark times, and the
oracle on sampled heads (rows and heads are independent, which the oracle's own
row-independence pin establishes)."""
import math

import numpy as np
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
import oracle
from metaplastic_linear_attention_gb300 import synthetic as syn
from tests._helpers import TIGHT, oracle_forward_from, pick, rel_l2, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu(inputs):
    return {k: v.to(DEV) for k, v in inputs.items()}


def _fwd(gi, mu0=None, I0=None, chunk=0, **kw):
    out = pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                       gi["I_prior"], mu0, I0, chunk=chunk, **kw)
    assert pal.palimpsa_get_device_status() == 0
    return out


def _check_all(out, ref, tol, tight=None):
    errs = [rel_l2(o.cpu().numpy(), r) for o, r in zip(out, ref)]
    assert max(errs) <= tol, errs
    if tight is not None:
        assert max(errs) <= tight, errs
    return errs


def _random_state(B, H, dv, dk, seed, I_lo=0.5, I_hi=4.0):
    g = torch.Generator().manual_seed(seed)
    mu0 = torch.randn((B, H, dv, dk), generator=g)
    I0 = I_lo + (I_hi - I_lo) * torch.rand((B, H, dv, dk), generator=g)
    return mu0, I0


# ----------------------------------------------------------------- small, everything checked

def test_tiny_workload_all_chunks_bitwise_equal():
    """The fp32 tiny sequence (B=1, H=2, T=256, d=64): parity with the oracle, and
    the staging chunk size leaves the result bit-for-bit unchanged."""
    wl = syn.WORKLOADS["tiny"]
    inp = syn.sequence_inputs(wl)
    ref = oracle_forward_from(inp)
    gi = _gpu(inp)
    _check_all(_fwd(gi, chunk=wl.chunk), ref, tol_for(inp), TIGHT)   # automatic time split
    pal.palimpsa_set_forward_segments(1)                               # one segment: chunk is staging only
    try:
        outs = [_fwd(gi, chunk=c) for c in (16, 32, 64, 128)]
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check_all(outs[0], ref, tol_for(inp), TIGHT)
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a, b)


CASES = [
    # (B, H, T, d_k, d_v, bf16, chunk)
    (1, 1, 1, 128, 64, True, 16),
    (2, 3, 5, 128, 64, True, 32),
    (1, 2, 77, 64, 8, False, 16),
    (3, 2, 130, 128, 24, True, 64),
    (2, 1, 200, 64, 128, True, 32),
    (1, 3, 97, 128, 256, False, 16),
    (4, 5, 33, 128, 64, False, 32),
    (1, 1, 300, 64, 40, True, 64),
    (2, 2, 190, 128, 64, True, 128),
]


@pytest.mark.parametrize("B,H,T,dk,dv,bf16,chunk", CASES)
def test_forward_ragged_and_odd_shapes(B, H, T, dk, dv, bf16, chunk):
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16, chunk=chunk)
    inp = syn.sequence_inputs(wl, seed=1000 + T)
    ref = oracle_forward_from(inp)
    out = _fwd(_gpu(inp), chunk=chunk)
    _check_all(out, ref, tol_for(inp), TIGHT)


@pytest.mark.parametrize("bf16", [False, True])
def test_forward_initial_state_and_in_place(bf16):
    B, H, T, dk, dv = 2, 3, 150, 128, 64
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=7)
    mu0, I0 = _random_state(B, H, dv, dk, 8)
    ref = oracle_forward_from(inp, mu0=mu0, I0=I0)
    gi = _gpu(inp)
    out = _fwd(gi, mu0.to(DEV), I0.to(DEV))
    _check_all(out, ref, tol_for(inp), TIGHT)
    # in place: mu_T aliases mu0, I_T aliases I0
    m, i = mu0.to(DEV), I0.to(DEV)
    y, mT, IT = _fwd(gi, m, i, mu_T=m, I_T=i)
    assert mT.data_ptr() == m.data_ptr() and IT.data_ptr() == i.data_ptr()
    for a, b in zip((y, mT, IT), out):
        assert torch.equal(a, b)


def test_forward_empty_sequence_passes_state_through():
    B, H, dk, dv = 2, 2, 128, 64
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=0)
    inp = syn.sequence_inputs(wl)
    mu0, I0 = _random_state(B, H, dv, dk, 3)
    gi = _gpu(inp)
    y, mT, IT = _fwd(gi, mu0.to(DEV), I0.to(DEV))
    assert y.numel() == 0
    assert torch.equal(mT.cpu(), mu0) and torch.equal(IT.cpu(), I0)
    y, mT, IT = _fwd(gi)
    assert torch.all(mT == 0) and torch.equal(IT.cpu(), torch.ones_like(I0))


def test_forward_continuation_matches_single_pass():
    """Checkpoint/resume: the scan split at t = 70 and resumed from (mu_T, I_T)."""
    wl = syn.WORKLOADS["small_layer"].with_(B=2, H=2, T=200)
    inp = syn.sequence_inputs(wl, seed=11)
    gi = _gpu(inp)
    y, mT, IT = _fwd(gi)
    s = 70
    first = {k: (v[:, :, :s].contiguous() if v.dim() >= 3 else v) for k, v in gi.items()}
    second = {k: (v[:, :, s:].contiguous() if v.dim() >= 3 else v) for k, v in gi.items()}
    y1, m1, i1 = _fwd(first)
    y2, m2, i2 = _fwd(second, m1, i1)
    # The two runs split time differently; a split's segment summaries come from
    # the tensor cores with operands split into two bf16 parts (at most 2^-18
    # relative per product), so the runs agree to ~1e-6, not to fp32 rounding.
    assert rel_l2(torch.cat([y1, y2], 2).cpu(), y.cpu()) < 1e-5
    assert rel_l2(m2.cpu(), mT.cpu()) < 1e-5 and rel_l2(i2.cpu(), IT.cpu()) < 1e-5


# ----------------------------------------------------------------- decode step

STEP_CASES = [(1, 1, 128, 64, True), (3, 5, 128, 64, False), (2, 3, 64, 8, True), (4, 2, 64, 24, False),
              (2, 2, 128, 256, True), (5, 3, 128, 40, True)]


@pytest.mark.parametrize("B,H,dk,dv,bf16", STEP_CASES)
def test_step_matches_oracle_over_several_tokens(B, H, dk, dv, bf16):
    wl = syn.WORKLOADS["decode"].with_(B=B, H=H, d_k=dk, d_v=dv, bf16=bf16)
    seq = syn.sequence_inputs(wl, T=1, seed=5)
    steps = syn.decode_inputs(wl, 6, seed=5)
    mu0, I0 = _random_state(B, H, dv, dk, 9)
    mu, I = mu0.to(DEV).clone(), I0.to(DEV).clone()
    A, Ip = seq["A"].to(DEV), seq["I_prior"].to(DEV)
    rmu, rI = mu0.double().numpy(), I0.double().numpy()
    import oracle
    for s in range(6):
        gs = {k: v[s].to(DEV) for k, v in steps.items()}
        y = pal.palimpsa_step(gs["q"], gs["k"], gs["v"], gs["beta"], gs["d_t"], A, Ip, mu, I)
        f = syn.as_float64_numpy
        ry, rmu, rI = oracle.step(f(steps["q"][s]), f(steps["k"][s]), f(steps["v"][s]), f(steps["beta"][s]),
                                  f(steps["d_t"][s]), f(seq["A"]), f(seq["I_prior"]), rmu, rI)
        assert rel_l2(y.cpu(), ry) <= TIGHT
    assert pal.palimpsa_get_device_status() == 0
    assert rel_l2(mu.cpu(), rmu) <= TIGHT and rel_l2(I.cpu(), rI) <= TIGHT


def test_step_equals_one_token_forward():
    wl = syn.WORKLOADS["small_layer"].with_(B=3, H=4, T=1)
    inp = _gpu(syn.sequence_inputs(wl, seed=21))
    mu0, I0 = (t.to(DEV) for t in _random_state(3, 4, 64, 128, 22))
    y_f, m_f, i_f = _fwd(inp, mu0, I0)
    mu, I = mu0.clone(), I0.clone()
    y_s = pal.palimpsa_step(inp["q"][:, :, 0].contiguous(), inp["k"][:, :, 0].contiguous(),
                            inp["v"][:, :, 0].contiguous(), inp["beta"][:, :, 0].contiguous(),
                            inp["d_t"][:, :, 0].contiguous(), inp["A"], inp["I_prior"], mu, I)
    assert rel_l2(y_s.cpu(), y_f[:, :, 0].cpu()) < 1e-6
    assert rel_l2(mu.cpu(), m_f.cpu()) < 1e-6 and torch.allclose(I, i_f, rtol=1e-6)


# ----------------------------------------------------------------- full-size workloads

def test_small_layer_full_size():
    """B=4, H=16, T=2048, d_k=128, d_v=64, bf16: every output against the oracle."""
    wl = syn.WORKLOADS["small_layer"]
    inp = syn.sequence_inputs(wl)
    out = _fwd(_gpu(inp), chunk=wl.chunk)
    ref = oracle_forward_from(inp)
    _check_all(out, ref, tol_for(inp), TIGHT)


@pytest.mark.parametrize("name", ["layer_760m", "long_context"])
def test_large_workloads_every_head(name):
    """Full-size launches in the benchmark's configuration (automatic time split);
    the oracle recomputes every head over all T tokens (192 heads x 4096 tokens,
    32 heads x 32768 tokens: seconds of fp64 work on the host cores)."""
    wl = syn.WORKLOADS[name]
    plan = pal.palimpsa_forward_plan(wl.B, wl.H, wl.T, wl.d_k, wl.d_v, chunk=wl.chunk, bf16=wl.bf16)
    assert plan["segments"] > 1          # the launch under test is the split one
    inp = syn.sequence_inputs(wl)
    out = _fwd(_gpu(inp), chunk=wl.chunk)
    ref = oracle_forward_from(inp)
    _check_all(out, ref, tol_for(inp), TIGHT)
    # per head as well: no head may hide behind the others' norm
    y, _, IT = out
    yn = y.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            assert rel_l2(yn[b, h], ref[0][b, h]) <= TIGHT, (b, h)
    assert (IT > 0).all()


def test_decode_workload_prefill_and_steps_sampled_heads():
    """B=256, H=32: the 512-token prefill then decode steps one call per token;
    sampled heads replayed by the oracle's single-token step function."""
    wl = syn.WORKLOADS["decode"]
    S = 8
    inp = syn.sequence_inputs(wl)
    steps = syn.decode_inputs(wl, S)
    gi = _gpu(inp)
    _, mu, I = _fwd(gi, chunk=wl.chunk)
    heads = [(0, 0), (17, 5), (128, 31), (255, 16)]
    _, rmu, rI = oracle_forward_from(inp, heads=heads)
    bs = [b for b, _ in heads]
    hs = [h for _, h in heads]
    f = syn.as_float64_numpy
    for s in range(S):
        gs = {k: v[s].to(DEV) for k, v in steps.items()}
        y = pal.palimpsa_step(gs["q"], gs["k"], gs["v"], gs["beta"], gs["d_t"], gi["A"], gi["I_prior"], mu, I)
        sel = {k: f(v[s])[bs, hs][None] for k, v in steps.items()}
        ry, rmu, rI = oracle.step(sel["q"], sel["k"], sel["v"], sel["beta"], sel["d_t"],
                                  f(inp["A"])[hs], f(inp["I_prior"])[hs], rmu, rI)
        assert rel_l2(pick(y, heads), ry) <= TIGHT
    assert pal.palimpsa_get_device_status() == 0
    assert rel_l2(pick(mu, heads), rmu) <= TIGHT and rel_l2(pick(I, heads), rI) <= TIGHT


def test_decode_job_every_step_every_head():
    """The whole decode job exactly as the benchmark launches it: B=256, H=32,
    d_k=128, d_v=64, bf16 inputs made on the device with the benchmark's seed; the
    512-token prefill, then one palimpsa_step call over all 1024 decode tokens (one
    step sequence: alternating walks, the default L2 hand-over between steps,
    dependent launches). The oracle runs each head as one continuous scan of
    512 + 1024 tokens (a decode step is one token of the recurrence), on every
    head, in groups of batch rows; y of every decode step, the prefill's y and
    the final mu, I are compared."""
    wl = syn.WORKLOADS["decode"]
    B, H, T, S, dv = wl.B, wl.H, wl.T, wl.steps, wl.d_v
    assert S == 1024
    inp = syn.sequence_inputs(wl, device=DEV)
    dec = syn.decode_inputs(wl, S, device=DEV)
    y_pre, mu, I = _fwd(inp, chunk=wl.chunk)
    y_dec = pal.palimpsa_step(dec["q"], dec["k"], dec["v"], dec["beta"], dec["d_t"], inp["A"], inp["I_prior"],
                              mu, I)
    torch.cuda.synchronize()
    assert pal.palimpsa_get_device_status() == 0
    f = syn.as_float64_numpy
    A, Ip = f(inp["A"]), f(inp["I_prior"])
    y_dec_h = y_dec.cpu()                                   # [S, B, H, dv]
    err_steps = np.zeros((S, 2))                            # per step: sum |diff|^2, sum |ref|^2
    err_pre, err_mu, err_I = np.zeros(2), np.zeros(2), np.zeros(2)
    G = 16                                                  # batch rows per oracle call (512 heads)
    for b0 in range(0, B, G):
        b1 = b0 + G
        seq = {}
        for n in ("q", "k", "v", "beta", "d_t"):
            steps_n = dec[n][:, b0:b1].movedim(0, 2)        # [G, H, S, ...]
            seq[n] = f(torch.cat([inp[n][b0:b1].float(), steps_n.float()], dim=2))
        ry, rmu, rI = oracle.forward(seq["q"], seq["k"], seq["v"], seq["beta"], seq["d_t"], A, Ip)
        gy = y_dec_h[:, b0:b1].double().numpy()             # [S, G, H, dv]
        ref_steps = np.moveaxis(ry[:, :, T:], 2, 0)         # [S, G, H, dv]
        err_steps[:, 0] += ((gy - ref_steps) ** 2).reshape(S, -1).sum(1)
        err_steps[:, 1] += (ref_steps ** 2).reshape(S, -1).sum(1)
        for acc, got, ref in ((err_pre, y_pre[b0:b1], ry[:, :, :T]), (err_mu, mu[b0:b1], rmu),
                              (err_I, I[b0:b1], rI)):
            g = f(got)
            acc += (((g - ref) ** 2).sum(), (ref ** 2).sum())
    step_err = np.sqrt(err_steps[:, 0] / err_steps[:, 1])
    assert step_err.max() <= TIGHT, (int(step_err.argmax()), float(step_err.max()))
    for name, acc in (("prefill y", err_pre), ("mu", err_mu), ("I", err_I)):
        assert np.sqrt(acc[0] / acc[1]) <= TIGHT, name


# ----------------------------------------------------------------- failure detection (no fault)

def test_domain_violation_is_reported_not_faulted():
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=40)
    gi = _gpu(syn.sequence_inputs(wl))
    gi["A"] = gi["A"].clone()
    gi["A"][1] = -1.0
    pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"])
    assert pal.palimpsa_get_device_status() == 5          # PALIMPSA_ERR_DOMAIN
    assert pal.palimpsa_get_device_status() == 0          # read-and-clear
    gi["A"][1] = 0.5
    _fwd(gi)


@pytest.mark.parametrize("what", ["beta", "d_t", "A", "I_prior", "I0"])
def test_backward_domain_violation_is_reported_not_faulted(what):
    """The backward reports a broken precondition of its inputs (beta >= 0, d_t >= 0,
    A > 0, I_prior > 0, I0 > 0) as PALIMPSA_ERR_DOMAIN without a fault; the next
    call is clean."""
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=70)
    gi = _gpu(syn.sequence_inputs(wl))
    mu0, I0 = (t.to(DEV) for t in _random_state(1, 2, wl.d_v, wl.d_k, 11))
    dy = torch.randn((1, 2, 70, wl.d_v), device=DEV)
    bad = {k: v.clone() for k, v in gi.items()}
    bad_I0 = I0.clone()
    if what == "beta":
        bad["beta"][0, 1, 37, 5] = -0.5
    elif what == "d_t":
        bad["d_t"][0, 0, 3] = -1.0
    elif what == "A":
        bad["A"][1] = -0.5
    elif what == "I_prior":
        bad["I_prior"][0] = 0.0
    else:
        bad_I0[0, 1, 3, 7] = -2.0
    pal.palimpsa_backward(bad["q"], bad["k"], bad["v"], bad["beta"], bad["d_t"], bad["A"], bad["I_prior"], mu0,
                          bad_I0, dy)
    assert pal.palimpsa_get_device_status() == 5          # PALIMPSA_ERR_DOMAIN
    pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], mu0, I0, dy)
    assert pal.palimpsa_get_device_status() == 0


@pytest.mark.parametrize("what", ["beta", "d_t", "A"])
def test_segment_summary_domain_violation_is_reported_not_faulted(what):
    """The segment summary reports a broken precondition of its inputs (checked before pass A)."""
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=300)
    gi = _gpu(syn.sequence_inputs(wl))
    bad = {k: v.clone() for k, v in gi.items()}
    if what == "beta":
        bad["beta"][0, 0, 200, 9] = -1.0
    elif what == "d_t":
        bad["d_t"][0, 1, 17] = float("nan")
    else:
        bad["A"][0] = 0.0
    pal.palimpsa_set_forward_segments(3)
    try:
        pal.palimpsa_segment_summary(bad["q"], bad["k"], bad["v"], bad["beta"], bad["d_t"], bad["A"],
                                     bad["I_prior"])
        assert pal.palimpsa_get_device_status() == 5      # PALIMPSA_ERR_DOMAIN
        pal.palimpsa_segment_summary(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"])
        assert pal.palimpsa_get_device_status() == 0
    finally:
        pal.palimpsa_set_forward_segments(0)


@pytest.mark.parametrize("S", [1, 3])
def test_withheld_copy_times_out_and_context_survives(S):
    """A staged copy that never arrives: the bounded mbarrier wait gives up, the
    kernel latches PALIMPSA_ERR_TIMEOUT and returns; later calls work. With S = 3
    the tensor-core summary kernel times out first: it must drain and free its
    tensor memory, or the next call's summaries could not allocate any."""
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=100)
    inp = syn.sequence_inputs(wl)
    gi = _gpu(inp)
    pal.palimpsa_set_wait_timeout_ns(2_000_000)
    pal.palimpsa_set_forward_segments(S)
    pal.palimpsa_debug_withhold_first_copy(True)
    try:
        pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                     gi["I_prior"], chunk=32)
        assert pal.palimpsa_get_device_status() == 8       # PALIMPSA_ERR_TIMEOUT
    finally:
        pal.palimpsa_debug_withhold_first_copy(False)
        pal.palimpsa_set_wait_timeout_ns(2_000_000_000)
    try:
        out = _fwd(gi, chunk=32)
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check_all(out, oracle_forward_from(inp), tol_for(inp), TIGHT)


def test_host_buffers_end_to_end():
    """The public call with pinned host tensors copies in, computes on the GPU and copies out."""
    wl = syn.WORKLOADS["small_layer"].with_(B=2, H=2, T=64)
    inp = {k: v.pin_memory() for k, v in syn.sequence_inputs(wl, seed=4).items()}
    y, mT, IT = pal.palimpsa_forward_chunked(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"],
                                             inp["I_prior"])
    assert y.device.type == "cpu"
    _check_all((y, mT, IT), oracle_forward_from(inp), tol_for(inp), TIGHT)


# ----------------------------------------------------------------- time split (segments)

SPLIT_CASES = [
    # (B, H, T, d_k, d_v, bf16, segments)
    (1, 2, 100, 128, 64, True, 2),
    (2, 1, 333, 128, 64, True, 3),
    (1, 3, 257, 64, 8, False, 7),
    (1, 1, 1000, 128, 24, True, 16),
    (2, 2, 64, 128, 128, False, 4),
    (1, 2, 17, 128, 64, True, 5),      # more segments requested than whole chunks exist
    # tensor-core summaries at each d_v they serve (TMEM columns 64 / 128 / 256)
    (1, 2, 300, 128, 32, True, 3),
    (1, 1, 500, 128, 96, True, 4),
    (2, 1, 400, 128, 128, True, 5),
]


@pytest.mark.parametrize("B,H,T,dk,dv,bf16,S", SPLIT_CASES)
def test_time_split_matches_oracle(B, H, T, dk, dv, bf16, S):
    """Segment summaries + carry + per-segment recurrence equal the sequential scan."""
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=3000 + T)
    mu0, I0 = _random_state(B, H, dv, dk, 31)
    ref = oracle_forward_from(inp, mu0=mu0, I0=I0)
    gi = _gpu(inp)
    pal.palimpsa_set_forward_segments(S)
    try:
        out = _fwd(gi, mu0.to(DEV), I0.to(DEV), chunk=16)
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check_all(out, ref, tol_for(inp), TIGHT)
    unsplit = _fwd(gi, mu0.to(DEV), I0.to(DEV), chunk=16)
    # bf16 summaries come from the tensor cores (two-part bf16 operands, at most
    # 2^-18 relative per product), fp32 ones from FFMA
    for a, b in zip(out, unsplit):
        assert rel_l2(a.cpu(), b.cpu()) < (1e-5 if bf16 else 1e-6)


def test_time_split_with_default_state_and_in_place():
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=300)
    inp = syn.sequence_inputs(wl, seed=77)
    gi = _gpu(inp)
    ref = oracle_forward_from(inp)
    pal.palimpsa_set_forward_segments(6)
    try:
        out = _fwd(gi, chunk=32)
        _check_all(out, ref, tol_for(inp), TIGHT)
        mu0, I0 = _random_state(1, 2, 64, 128, 78)
        m, i = mu0.to(DEV), I0.to(DEV)
        y, mT, IT = _fwd(gi, m, i, mu_T=m, I_T=i, chunk=32)
        _check_all((y, mT, IT), oracle_forward_from(inp, mu0=mu0, I0=I0), tol_for(inp), TIGHT)
    finally:
        pal.palimpsa_set_forward_segments(0)


# ----------------------------------------------------------------- host buffers, pipelined

def test_host_forward_pipeline_matches_device_path(monkeypatch):
    """Pinned host inputs streamed in several batch blocks give the device path's results."""
    import metaplastic_linear_attention_gb300.binding as b
    wl = syn.WORKLOADS["small_layer"].with_(B=5, H=3, T=96)
    inp = syn.sequence_inputs(wl, seed=61)
    g = torch.Generator().manual_seed(62)
    mu0 = torch.randn((5, 3, 64, 128), generator=g)
    I0 = 0.5 + torch.rand((5, 3, 64, 128), generator=g)
    ref = _fwd(_gpu(inp), mu0.to(DEV), I0.to(DEV))
    monkeypatch.setattr(b, "HOST_BLOCK_BYTES", 1)          # one batch entry per block: 5 blocks
    monkeypatch.setattr(b, "MIN_HEADS_PER_FORWARD_BLOCK", 1)
    host = {k: v.pin_memory() for k, v in inp.items()}
    y, mT, IT = pal.palimpsa_forward_chunked(host["q"], host["k"], host["v"], host["beta"], host["d_t"], host["A"],
                                             host["I_prior"], mu0.pin_memory(), I0.pin_memory())
    assert y.device.type == "cpu" and mT.device.type == "cpu"
    # 3-head blocks may be planned with other time splits than the 15-head call, and
    # bf16 segment summaries agree to ~1e-6 across splits (tensor-core operands)
    for a_, r_ in zip((y, mT, IT), ref):
        assert rel_l2(a_, r_.cpu()) < 1e-5
    # state outputs on the device, y to the host
    m_d, i_d = torch.empty_like(mu0, device=DEV), torch.empty_like(I0, device=DEV)
    y2, m2, i2 = pal.palimpsa_forward_chunked(host["q"], host["k"], host["v"], host["beta"], host["d_t"], host["A"],
                                              host["I_prior"], y=torch.empty_like(y).pin_memory(), mu_T=m_d, I_T=i_d)
    assert m2.data_ptr() == m_d.data_ptr() and y2.device.type == "cpu"
    ref_default = _fwd(_gpu(inp))
    assert rel_l2(y2, ref_default[0].cpu()) < 1e-5 and rel_l2(m2.cpu(), ref_default[1].cpu()) < 1e-5


def test_step_sequence_host_pipeline_matches_token_by_token(monkeypatch):
    import metaplastic_linear_attention_gb300.binding as b
    wl = syn.WORKLOADS["decode"].with_(B=4, H=3)
    seq = syn.sequence_inputs(wl, T=1, seed=71)
    steps = syn.decode_inputs(wl, 11, seed=71)
    mu0, I0 = _random_state(4, 3, 64, 128, 72)
    A, Ip = seq["A"].to(DEV), seq["I_prior"].to(DEV)
    mu, I = mu0.to(DEV), I0.to(DEV)
    ys = [pal.palimpsa_step(*(steps[n][t].to(DEV) for n in ("q", "k", "v", "beta", "d_t")), A, Ip, mu, I).cpu()
          for t in range(11)]
    monkeypatch.setattr(b, "HOST_BLOCK_BYTES", 1)          # one token per block: 11 blocks
    mu2, I2 = mu0.to(DEV), I0.to(DEV)
    host = {k: v.pin_memory() for k, v in steps.items()}
    y = pal.palimpsa_step(host["q"], host["k"], host["v"], host["beta"], host["d_t"], seq["A"], seq["I_prior"],
                          mu2, I2)
    assert y.shape == (11, 4, 3, 64) and y.device.type == "cpu"
    assert torch.equal(y, torch.stack(ys))
    assert torch.equal(mu2, mu) and torch.equal(I2, I)
    # device-resident sequence
    mu3, I3 = mu0.to(DEV), I0.to(DEV)
    y3 = pal.palimpsa_step(*(steps[n].to(DEV) for n in ("q", "k", "v", "beta", "d_t")), A, Ip, mu3, I3)
    assert torch.equal(y3.cpu(), y) and torch.equal(mu3, mu)


# ----------------------------------------------------------------- "without Meta" comparator

@pytest.mark.parametrize("S", [0, 1, 3])
@pytest.mark.parametrize("B,H,T,dk,dv,bf16", [(1, 2, 1, 128, 64, True), (2, 3, 77, 128, 64, True),
                                              (1, 2, 130, 64, 24, False), (3, 1, 200, 128, 128, False)])
def test_without_meta_matches_oracle(B, H, T, dk, dv, bf16, S):
    from oracle import reference_np as rnp
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=900 + T)
    g = torch.Generator().manual_seed(901)
    mu0 = torch.randn((B, H, dv, dk), generator=g)
    f = syn.as_float64_numpy
    ry, rmu = rnp.forward_without_meta(*(f(inp[n]) for n in ("q", "k", "v", "beta", "d_t", "A", "I_prior")),
                                       mu0=f(mu0))
    gi = _gpu(inp)
    m = mu0.to(DEV)
    pal.palimpsa_set_forward_segments(S)   # 0: the forward's automatic plan
    try:
        y, mT = pal.palimpsa_forward_without_meta(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                                  gi["I_prior"], m, mu_T=m)   # in place
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0
    assert rel_l2(y.cpu(), ry) <= TIGHT and rel_l2(mT.cpu(), rmu) <= TIGHT


def test_without_meta_full_size_sampled_heads():
    from oracle import reference_np as rnp
    wl = syn.WORKLOADS["layer_760m"]
    inp = syn.sequence_inputs(wl)
    gi = _gpu(inp)
    y, mT = pal.palimpsa_forward_without_meta(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                              gi["I_prior"])
    assert pal.palimpsa_get_device_status() == 0
    heads = [(0, 0), (6, 19)]
    bs, hs = [b for b, _ in heads], [h for _, h in heads]
    f = syn.as_float64_numpy
    sel = [f(inp[n])[bs, hs][None] for n in ("q", "k", "v", "beta", "d_t")]
    ry, rmu = rnp.forward_without_meta(*sel, f(inp["A"])[hs], f(inp["I_prior"])[hs])
    assert rel_l2(pick(y, heads), ry) <= TIGHT and rel_l2(pick(mT, heads), rmu) <= TIGHT


# ----------------------------------------------------------------- backward

BWD_CASES = [
    # (B, H, T, d_k, d_v, bf16, with_state, with_final_grads)
    (1, 2, 100, 128, 64, False, True, True),
    (2, 1, 70, 128, 64, True, False, False),
    (1, 2, 9, 64, 8, False, True, False),
    (1, 1, 1, 128, 16, True, False, True),
    (1, 1, 200, 128, 64, True, True, True),
]


def _bwd_case(B, H, T, dk, dv, bf16, with_state, with_final, seed):
    from oracle import autograd as ag
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    mu0 = torch.randn((B, H, dv, dk), generator=g) if with_state else None
    I0 = (0.5 + 2.0 * torch.rand((B, H, dv, dk), generator=g)) if with_state else None
    dy = torch.randn((B, H, T, dv), generator=g)
    dmu = torch.randn((B, H, dv, dk), generator=g) if with_final else None
    dI = torch.randn((B, H, dv, dk), generator=g) if with_final else None
    f = syn.as_float64_numpy
    ref = ag.gradients({n: (None if t is None else f(t)) for n, t in
                        dict(q=inp["q"], k=inp["k"], v=inp["v"], beta=inp["beta"], d_t=inp["d_t"], A=inp["A"],
                             I_prior=inp["I_prior"], mu0=mu0, I0=I0).items()},
                       f(dy), None if dmu is None else f(dmu), None if dI is None else f(dI))
    d = lambda t: None if t is None else t.to(DEV)
    gi = _gpu(inp)
    out = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], d(mu0),
                                d(I0), d(dy), d(dmu), d(dI))
    assert pal.palimpsa_get_device_status() == 0
    return out, ref, with_state


@pytest.mark.parametrize("B,H,T,dk,dv,bf16,with_state,with_final", BWD_CASES)
def test_backward_matches_fp64_autograd(B, H, T, dk, dv, bf16, with_state, with_final):
    out, ref, with_state = _bwd_case(B, H, T, dk, dv, bf16, with_state, with_final, seed=4000 + T)
    pairs = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t"), ("dA", "A"),
             ("dI_prior", "I_prior")]
    if with_state:
        pairs += [("dmu0", "mu0"), ("dI0", "I0")]
    errs = {n: rel_l2(out[n].cpu(), ref[m]) for n, m in pairs}
    assert max(errs.values()) <= TIGHT, errs


def test_backward_empty_sequence():
    out, ref, _ = _bwd_case(1, 2, 0, 128, 64, False, True, True, seed=4500)
    assert rel_l2(out["dmu0"].cpu(), ref["mu0"]) <= 1e-6 and rel_l2(out["dI0"].cpu(), ref["I0"]) <= 1e-6
    assert rel_l2(out["dI_prior"].cpu(), ref["I_prior"]) <= 1e-6 or float(abs(out["dI_prior"]).max()) == 0.0


def test_forward_plan_reports_the_split():
    """palimpsa_forward_plan: many heads run unsplit in one launch; few long heads are
    split into segments (three launches) with scratch per boundary; a forced count is
    honoured."""
    wide = pal.palimpsa_forward_plan(256, 32, 512, 128, 64)
    assert wide["segments"] == 1 and wide["launches"] == 1 and wide["scratch_bytes"] == 0
    few = pal.palimpsa_forward_plan(1, 32, 32768, 128, 64)
    assert few["segments"] > 1 and few["launches"] == 3
    b = few["segments"] - 1                                    # boundaries
    states, gammas, init = 32 * b * 2 * 64 * 128, 32 * b, 32 * 2 * 64 * 128
    assert few["scratch_bytes"] == 4 * ((states + gammas + 3) // 4 * 4 + init)
    assert few["segment_len"] * few["segments"] >= 32768 > few["segment_len"] * (few["segments"] - 1)
    pal.palimpsa_set_forward_segments(4)
    try:
        assert pal.palimpsa_forward_plan(2, 3, 1000, 128, 64)["segments"] == 4
    finally:
        pal.palimpsa_set_forward_segments(0)


# ----------------------------------------------------------------- extreme gates and states

def _extreme_inputs(bf16, seed):
    """Gates at both ends (alpha = 1 exactly, alpha underflowing to 0, and values in
    between), beta zero on whole tokens and rows, initial precisions over six
    orders of magnitude."""
    B, H, T, dk, dv = 2, 2, 150, 128, 64
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=seed)
    g = torch.Generator().manual_seed(seed)
    pick_dt = torch.tensor([0.0, 1e-4, 0.05, 1.0, 30.0, 500.0])
    inp["d_t"] = pick_dt[torch.randint(0, len(pick_dt), (B, H, T), generator=g)].contiguous()
    beta = inp["beta"].float()
    beta[:, :, ::7] = 0.0                   # tokens that write nothing
    beta[:, :, :, ::5] = 0.0                # value rows that never learn
    inp["beta"] = beta.to(inp["beta"].dtype).contiguous()
    mu0 = torch.randn((B, H, dv, dk), generator=g)
    I0 = 10.0 ** (6.0 * torch.rand((B, H, dv, dk), generator=g) - 3.0)   # 1e-3 .. 1e3
    return inp, mu0, I0


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("S", [1, 3])
def test_forward_extreme_gates_and_states(bf16, S):
    inp, mu0, I0 = _extreme_inputs(bf16, 4100 + S)
    ref = oracle_forward_from(inp, mu0=mu0, I0=I0)
    pal.palimpsa_set_forward_segments(S)
    try:
        out = _fwd(_gpu(inp), mu0.to(DEV), I0.to(DEV))
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check_all(out, ref, tol_for(inp), TIGHT)


def test_step_extreme_gates_and_states():
    inp, mu0, I0 = _extreme_inputs(True, 4200)
    gi = _gpu(inp)
    mu, I = mu0.to(DEV), I0.to(DEV)
    f = syn.as_float64_numpy
    mu_r, I_r = f(mu0), f(I0)
    import oracle
    for t in range(12):
        tok = {k: (gi[k][:, :, t].contiguous() if gi[k].dim() >= 3 else gi[k]) for k in ("q", "k", "v", "beta", "d_t")}
        y = pal.palimpsa_step(tok["q"], tok["k"], tok["v"], tok["beta"], tok["d_t"], gi["A"], gi["I_prior"], mu, I)
        y_r, mu_r, I_r = oracle.step(*(f(inp[n][:, :, t]) for n in ("q", "k", "v", "beta", "d_t")),
                                     f(inp["A"]), f(inp["I_prior"]), mu_r, I_r)
        assert rel_l2(y.cpu().numpy(), y_r) <= TIGHT
    assert pal.palimpsa_get_device_status() == 0
    assert rel_l2(mu.cpu().numpy(), mu_r) <= TIGHT and rel_l2(I.cpu().numpy(), I_r) <= TIGHT


def test_backward_extreme_gates_and_states():
    from oracle import autograd as oag
    inp, mu0, I0 = _extreme_inputs(False, 4300)
    g = torch.Generator().manual_seed(4301)
    dy = torch.randn(inp["q"].shape[:3] + (64,), generator=g)
    f = syn.as_float64_numpy
    ref = oag.gradients({n: f(t) for n, t in dict(q=inp["q"], k=inp["k"], v=inp["v"], beta=inp["beta"],
                                                  d_t=inp["d_t"], A=inp["A"], I_prior=inp["I_prior"],
                                                  mu0=mu0, I0=I0).items()}, f(dy))
    gi = _gpu(inp)
    got = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"],
                                mu0.to(DEV), I0.to(DEV), dy.to(DEV))
    assert pal.palimpsa_get_device_status() == 0
    errs = {n: rel_l2(got[n].cpu().numpy(), ref[n[1:]]) for n in
            ("dq", "dk", "dv", "dbeta", "dd_t", "dA", "dI_prior", "dmu0", "dI0")}
    assert max(errs.values()) <= TIGHT, errs


# ----------------------------------------------------------------- training checkpoints

@pytest.mark.parametrize("B,H,T,bf16,S", [(2, 2, 150, True, 1), (1, 2, 150, True, 3), (1, 3, 97, False, 1),
                                          (2, 1, 32, True, 1), (1, 1, 1, False, 1)])
def test_forward_checkpoints_are_the_states_every_32_tokens(B, H, T, bf16, S):
    """Checkpoint c holds (M, I) = (I mu, I) before token 32 c, as the oracle computes it."""
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=5000 + T + S)
    mu0, I0 = _random_state(B, H, 64, 128, 5001)
    gi = _gpu(inp)
    pal.palimpsa_set_forward_segments(S)
    try:
        y, mT, IT, ck = pal.palimpsa_forward_checkpointed(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                                          gi["I_prior"], mu0.to(DEV), I0.to(DEV))
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0
    _check_all((y, mT, IT), oracle_forward_from(inp, mu0=mu0, I0=I0), tol_for(inp), TIGHT)
    ck = ck.cpu().numpy()
    for c in range(ck.shape[2]):
        t = 32 * c
        if t == 0:
            mu_r, I_r = syn.as_float64_numpy(mu0), syn.as_float64_numpy(I0)
        else:
            prefix = {n: (x[:, :, :t].contiguous() if x.dim() >= 3 else x) for n, x in inp.items()}
            _, mu_r, I_r = oracle_forward_from(prefix, mu0=mu0, I0=I0)
        assert rel_l2(ck[:, :, c, :, 0, :], mu_r * I_r) <= TIGHT, c
        assert rel_l2(ck[:, :, c, :, 1, :], I_r) <= TIGHT, c


@pytest.mark.parametrize("B,H,T,dk,dv,bf16,with_state,with_final", [
    (2, 2, 150, 128, 64, True, True, True), (1, 3, 97, 64, 40, False, False, False),
    (1, 2, 1, 128, 64, True, True, False), (2, 1, 64, 128, 64, False, True, True)])
def test_backward_from_forward_checkpoints(B, H, T, dk, dv, bf16, with_state, with_final):
    """The backward reading the forward's checkpoints matches fp64 autograd, and the
    backward that recomputes its own checkpoints."""
    out, ref, _ = _bwd_case(B, H, T, dk, dv, bf16, with_state, with_final, seed=5100 + T)
    wl = syn.WORKLOADS["small_layer"].with_(B=B, H=H, T=T, d_k=dk, d_v=dv, bf16=bf16)
    inp = syn.sequence_inputs(wl, seed=5100 + T)
    g = torch.Generator().manual_seed(5100 + T + 1)
    mu0 = torch.randn((B, H, dv, dk), generator=g) if with_state else None
    I0 = (0.5 + 2.0 * torch.rand((B, H, dv, dk), generator=g)) if with_state else None
    dy = torch.randn((B, H, T, dv), generator=g)
    dmu = torch.randn((B, H, dv, dk), generator=g) if with_final else None
    dI = torch.randn((B, H, dv, dk), generator=g) if with_final else None
    d = lambda t: None if t is None else t.to(DEV)
    gi = _gpu(inp)
    _, _, _, ck = pal.palimpsa_forward_checkpointed(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                                    gi["I_prior"], d(mu0), d(I0))
    got = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], d(mu0),
                                d(I0), d(dy), d(dmu), d(dI), ckpt=ck)
    assert pal.palimpsa_get_device_status() == 0
    pairs = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t"), ("dA", "A"),
             ("dI_prior", "I_prior")] + ([("dmu0", "mu0"), ("dI0", "I0")] if with_state else [])
    errs = {n: rel_l2(got[n].cpu(), ref[m]) for n, m in pairs}
    assert max(errs.values()) <= TIGHT, errs
    same = {n: rel_l2(got[n].cpu(), out[n].cpu()) for n, _ in pairs}
    assert max(same.values()) <= 1e-5, same


def test_step_sequence_equals_token_by_token_bitwise():
    """One palimpsa_step_sequence call (4-D inputs on the device) enqueues the same
    launches as S palimpsa_step calls: identical bits."""
    wl = syn.WORKLOADS["decode"].with_(B=3, H=2)
    seq = _gpu(syn.sequence_inputs(wl, T=1, seed=81))
    steps = _gpu(syn.decode_inputs(wl, 9, seed=81))
    g = torch.Generator().manual_seed(82)
    mu0 = torch.randn((3, 2, 64, 128), generator=g).to(DEV)
    I0 = (0.5 + torch.rand((3, 2, 64, 128), generator=g)).to(DEV)
    mu_a, I_a = mu0.clone(), I0.clone()
    y_a = pal.palimpsa_step(steps["q"], steps["k"], steps["v"], steps["beta"], steps["d_t"], seq["A"],
                            seq["I_prior"], mu_a, I_a)
    mu_b, I_b = mu0.clone(), I0.clone()
    y_b = torch.stack([pal.palimpsa_step(steps["q"][t], steps["k"][t], steps["v"][t], steps["beta"][t],
                                         steps["d_t"][t], seq["A"], seq["I_prior"], mu_b, I_b) for t in range(9)])
    assert pal.palimpsa_get_device_status() == 0
    assert torch.equal(y_a, y_b) and torch.equal(mu_a, mu_b) and torch.equal(I_a, I_b)


@pytest.mark.parametrize("keep", [0, 128 << 10, 96 << 20])
def test_step_walk_order_and_l2_keep_change_no_bits(keep):
    """Decode steps walk the state in alternating orders and store the end of
    each walk with an L2-keeping policy. With the whole state kept, part of it or
    none (walk order fixed), the results are bit-identical to each other and
    match the oracle."""
    wl = syn.WORKLOADS["decode"].with_(B=6, H=4)
    seq = _gpu(syn.sequence_inputs(wl, T=1, seed=91))
    steps = _gpu(syn.decode_inputs(wl, 7, seed=91))
    g = torch.Generator().manual_seed(92)
    mu0 = torch.randn((6, 4, 64, 128), generator=g)
    I0 = 0.5 + torch.rand((6, 4, 64, 128), generator=g)

    def run(nbytes):
        pal.palimpsa_set_step_l2_keep_bytes(nbytes)
        try:
            mu, I = mu0.to(DEV), I0.to(DEV)
            y = pal.palimpsa_step(steps["q"], steps["k"], steps["v"], steps["beta"], steps["d_t"], seq["A"],
                                  seq["I_prior"], mu, I)
        finally:
            pal.palimpsa_set_step_l2_keep_bytes(96 << 20)
        assert pal.palimpsa_get_device_status() == 0
        return y.cpu(), mu.cpu(), I.cpu()

    ref = run(0)
    for _ in range(2):  # both walk directions come first once
        got = run(keep)
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
    f = syn.as_float64_numpy
    ys, mu_r, I_r = [], f(mu0), f(I0)
    for t in range(7):
        y_t, mu_r, I_r = oracle.forward(*(f(steps[n][t])[:, :, None] for n in ("q", "k", "v", "beta")),
                                        f(steps["d_t"][t])[:, :, None], f(seq["A"]), f(seq["I_prior"]),
                                        mu0=mu_r, I0=I_r)
        ys.append(y_t[:, :, 0])
    assert rel_l2(ref[0].numpy(), np.stack(ys)) <= TIGHT
    assert rel_l2(ref[1].numpy(), mu_r) <= TIGHT and rel_l2(ref[2].numpy(), I_r) <= TIGHT


def test_backward_full_size_small_layer_sampled_head():
    """The backward at the small layer's full size (B=4, H=16, T=2048, bf16), as the
    benchmark runs it, against fp64 autograd on one head across the whole batch:
    its per-token gradients, and dA, dI_prior of that head (sums over the batch)."""
    from oracle import autograd as ag
    wl = syn.WORKLOADS["small_layer"]
    inp = syn.sequence_inputs(wl)
    g = torch.Generator().manual_seed(4242)
    dy = torch.randn((wl.B, wl.H, wl.T, wl.d_v), generator=g)
    gi = _gpu(inp)
    out = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], None,
                                None, dy.to(DEV), want_state_grads=False)
    assert pal.palimpsa_get_device_status() == 0
    h = 5
    f = syn.as_float64_numpy
    sub = {n: f(inp[n][:, h:h + 1]) for n in ("q", "k", "v", "beta", "d_t")}
    sub.update(A=f(inp["A"][h:h + 1]), I_prior=f(inp["I_prior"][h:h + 1]), mu0=None, I0=None)
    ref = ag.gradients(sub, f(dy[:, h:h + 1]))
    for n, m in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t")):
        assert rel_l2(out[n][:, h:h + 1].cpu().numpy(), ref[m]) <= TIGHT, n
    for n, m in (("dA", "A"), ("dI_prior", "I_prior")):
        assert rel_l2(out[n][h:h + 1].cpu().numpy(), ref[m]) <= TIGHT, n


@pytest.mark.parametrize("name,b,h,r0", [("layer_760m", 7, 23, 60), ("long_context", 0, 17, 12)])
def test_backward_full_size_sampled_rows(name, b, h, r0):
    """The backward at the full size of the 760M layer (8 x 24 x 4096) and of the long
    context (32 x 32768, long memory), with the loss on four value rows of one
    sequence: rows are independent in Eq. (5), so every gradient of that loss is the
    fp64 autograd of the four-row problem, and all other rows, sequences and heads get
    exactly zero. dA (a sum over 4096 or 32768 tokens) is held through dd_t."""
    from oracle import autograd as ag
    from tests._helpers import dA_within_bar
    wl = syn.WORKLOADS[name]
    inp = syn.sequence_inputs(wl)
    rows = slice(r0, r0 + 4)
    g = torch.Generator().manual_seed(4343)
    dy = torch.zeros((wl.B, wl.H, wl.T, wl.d_v))
    dy[b, h, :, rows] = torch.randn((wl.T, 4), generator=g)
    gi = _gpu(inp)
    out = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], None,
                                None, dy.to(DEV), want_state_grads=False)
    assert pal.palimpsa_get_device_status() == 0
    f = syn.as_float64_numpy
    one = lambda t: f(t[b:b + 1, h:h + 1])
    sub = dict(q=one(inp["q"]), k=one(inp["k"]), v=one(inp["v"])[..., rows], beta=one(inp["beta"])[..., rows],
               d_t=one(inp["d_t"]), A=f(inp["A"][h:h + 1]), I_prior=f(inp["I_prior"][h:h + 1]), mu0=None, I0=None)
    ref = ag.gradients(sub, f(dy[b:b + 1, h:h + 1, :, rows]))
    for n, m in (("dq", "q"), ("dk", "k"), ("dd_t", "d_t")):
        assert rel_l2(out[n][b:b + 1, h:h + 1].cpu().numpy(), ref[m]) <= TIGHT, n
    for n, m in (("dv", "v"), ("dbeta", "beta")):
        assert rel_l2(out[n][b:b + 1, h:h + 1, :, rows].cpu().numpy(), ref[m]) <= TIGHT, n
    assert rel_l2(out["dI_prior"][h:h + 1].cpu().numpy(), ref["I_prior"]) <= TIGHT
    ok, detail = dA_within_bar(out["dA"][h:h + 1].cpu(), ref["A"], out["dd_t"][b:b + 1, h:h + 1].cpu(), ref["d_t"],
                               one(inp["d_t"]), f(inp["A"][h:h + 1]))
    assert ok, detail
    # nothing leaks into rows, sequences or heads without a loss
    mask = torch.zeros((wl.B, wl.H), dtype=torch.bool)
    mask[b, h] = True
    for n in ("dq", "dk", "dd_t"):
        assert not out[n][~mask.to(DEV)].any(), n
    for n in ("dv", "dbeta"):
        t = out[n].clone()
        t[b, h, :, rows] = 0
        assert not t.any(), n
    others = torch.ones(wl.H, dtype=torch.bool)
    others[h] = False
    assert not out["dA"][others.to(DEV)].any() and not out["dI_prior"][others.to(DEV)].any()


def test_host_inputs_on_a_side_stream():
    """Host inputs with a caller's stream: the copies in, the kernels and the
    copies out all run on that stream, so the results equal the device path's."""
    wl = syn.WORKLOADS["decode"].with_(B=4, H=3)
    seq = syn.sequence_inputs(wl, T=1, seed=97)
    tok = syn.decode_inputs(wl, 1, seed=97)
    g = torch.Generator().manual_seed(98)
    mu0 = torch.randn((4, 3, 64, 128), generator=g)
    I0 = 0.5 + torch.rand((4, 3, 64, 128), generator=g)
    args = [tok[n][0] for n in ("q", "k", "v", "beta", "d_t")] + [seq["A"], seq["I_prior"]]
    mu_d, I_d = mu0.to(DEV), I0.to(DEV)
    y_ref = pal.palimpsa_step(*[t.to(DEV) for t in args], mu_d, I_d).cpu()
    side = torch.cuda.Stream()
    mu_h, I_h = mu0.clone().pin_memory(), I0.clone().pin_memory()
    y = pal.palimpsa_step(*[t.pin_memory() for t in args], mu_h, I_h, stream=side)
    assert pal.palimpsa_get_device_status() == 0
    assert torch.equal(y, y_ref) and torch.equal(mu_h, mu_d.cpu()) and torch.equal(I_h, I_d.cpu())

    lengths = [50, 0, 77]
    wlv = syn.WORKLOADS["small_layer"].with_(seed=99)
    pk = syn.packed_inputs(wlv, lengths, H=2)
    d = {n: t.to(DEV) for n, t in pk.items() if n != "cu_seqlens"}
    ref = pal.palimpsa_forward_varlen(d["q"], d["k"], d["v"], d["beta"], d["d_t"], d["A"], d["I_prior"],
                                      pk["cu_seqlens"].to(DEV))
    out = pal.palimpsa_forward_varlen(d["q"], d["k"], d["v"], d["beta"], d["d_t"], d["A"], d["I_prior"],
                                      pk["cu_seqlens"], max_seqlen=77, stream=side)
    side.synchronize()
    assert pal.palimpsa_get_device_status() == 0
    assert all(torch.equal(a, b) for a, b in zip(out, ref))
