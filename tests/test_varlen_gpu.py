"""GPU parity of the packed variable-length forward (palimpsa_forward_varlen)
against the fp64 oracle, which runs each sequence on its own.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 7 / Eq. (5) per sequence, slide 9 (the state
carried along a sequence, and across segments by the affine scan)."""
import numpy as np
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import synthetic as syn
from metaplastic_linear_attention_gb300.synthetic import as_float64_numpy as f64
from oracle import varlen as ovl
from tests._helpers import TIGHT, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(lengths, H, dk, dv, bf16, seed):
    wl = syn.WORKLOADS["small_layer"].with_(d_k=dk, d_v=dv, bf16=bf16, seed=seed)
    return syn.packed_inputs(wl, lengths, H=H)


def _oracle(inp, mu0=None, I0=None):
    return ovl.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["beta"]), f64(inp["d_t"]),
                       f64(inp["A"]), f64(inp["I_prior"]), inp["cu_seqlens"].tolist(),
                       mu0=None if mu0 is None else f64(mu0), I0=None if I0 is None else f64(I0))


def _gpu(inp, mu0=None, I0=None, chunk=0, **kw):
    g = {k: v.to(DEV) for k, v in inp.items()}
    out = pal.palimpsa_forward_varlen(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"], g["I_prior"],
                                      g["cu_seqlens"], None if mu0 is None else mu0.to(DEV),
                                      None if I0 is None else I0.to(DEV), chunk=chunk, **kw)
    assert pal.palimpsa_get_device_status() == 0
    return out


def _check(out, ref):
    errs = [rel_l2(o.cpu().numpy(), r) for o, r in zip(out, ref)]
    assert max(errs) <= TIGHT, errs


CASES = [
    # (lengths, H, d_k, d_v, bf16, chunk, segments)
    ([1], 2, 128, 64, True, 16, 0),
    ([5, 0, 17, 1, 64], 3, 128, 64, True, 32, 0),
    ([130, 7, 0, 0, 61], 2, 64, 40, False, 16, 0),
    ([300, 45, 1, 199], 2, 128, 64, True, 32, 3),   # forced time split on a ragged mix
    ([0, 257, 96], 1, 64, 128, False, 16, 4),
    ([700, 3], 2, 128, 256, False, 32, 0),
]


@pytest.mark.parametrize("lengths,H,dk,dv,bf16,chunk,S", CASES)
def test_varlen_matches_oracle(lengths, H, dk, dv, bf16, chunk, S):
    inp = _inputs(lengths, H, dk, dv, bf16, seed=len(lengths) * 31 + dk + dv)
    ref = _oracle(inp)
    pal.palimpsa_set_forward_segments(S)
    try:
        out = _gpu(inp, chunk=chunk)
    finally:
        pal.palimpsa_set_forward_segments(0)
    _check(out, ref)


@pytest.mark.parametrize("S", [1, 3])
def test_varlen_initial_state_and_in_place(S):
    lengths = [40, 0, 211, 9]
    N, H, dk, dv = len(lengths), 2, 128, 64
    inp = _inputs(lengths, H, dk, dv, True, seed=8)
    g = torch.Generator().manual_seed(3)
    mu0 = torch.randn((N, H, dv, dk), generator=g)
    I0 = 0.5 + 3.0 * torch.rand((N, H, dv, dk), generator=g)
    ref = _oracle(inp, mu0, I0)
    gi = {k: v.to(DEV) for k, v in inp.items()}
    mu, I = mu0.to(DEV), I0.to(DEV)
    pal.palimpsa_set_forward_segments(S)
    try:
        y, _, _ = pal.palimpsa_forward_varlen(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"],
                                              gi["I_prior"], gi["cu_seqlens"], mu, I, mu_T=mu, I_T=I)
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0
    _check((y, mu, I), ref)


def test_varlen_equal_lengths_equal_the_dense_forward_bitwise():
    """Same plan, same kernels: N equal sequences give the dense batch's bits."""
    N, H, T = 3, 2, 150
    inp = _inputs([T] * N, H, 128, 64, True, seed=12)
    yv, mv, Iv = _gpu(inp)
    dense = lambda x: x.reshape((H, N, T) + x.shape[2:]).transpose(0, 1).contiguous()
    g = {k: dense(inp[k]).to(DEV) for k in ("q", "k", "v", "beta", "d_t")}
    yd, md, Id = pal.palimpsa_forward_chunked(g["q"], g["k"], g["v"], g["beta"], g["d_t"], inp["A"].to(DEV),
                                              inp["I_prior"].to(DEV))
    assert torch.equal(dense(yv.cpu()), yd.cpu())
    assert torch.equal(mv, md) and torch.equal(Iv, Id)


def test_varlen_long_and_short_mix_uses_the_time_split():
    """A few heads, one long sequence and short ones: the planner splits time."""
    lengths = [4000, 13, 250, 1]
    inp = _inputs(lengths, 2, 128, 64, True, seed=21)
    _check(_gpu(inp), _oracle(inp))


def test_bad_offsets_are_reported_not_faulted():
    """Offsets out of order, past total_T or longer than max_seqlen: the CTAs of
    that sequence read nothing, the call latches a domain error, and the other
    sequences and the context are unaffected."""
    lengths = [20, 30, 10]
    inp = _inputs(lengths, 2, 128, 64, True, seed=5)
    ref = _oracle(inp)
    g = {k: v.to(DEV) for k, v in inp.items()}
    total = sum(lengths)
    for cu in ([0, 20, 15, 60], [0, 20, 50, total + 40], [0, 20, 50, 60]):
        cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
        y, mu, I = pal.palimpsa_forward_varlen(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"], g["I_prior"],
                                               cu_d, max_seqlen=25)
        assert pal.palimpsa_get_device_status() == 5  # PALIMPSA_ERR_DOMAIN
        # sequence 0 ([0, 20), within max_seqlen) is still right
        assert rel_l2(y[:, :20].cpu().numpy(), ref[0][:, :20]) <= TIGHT
        assert rel_l2(mu[0].cpu().numpy(), ref[1][0]) <= TIGHT
    _check(_gpu(inp), ref)


@pytest.mark.parametrize("flags", [dict(qk_norm=True, v_star=False), dict(qk_norm=True, v_star=True),
                                   dict(qk_norm=False, v_star=True)])
@pytest.mark.parametrize("S", [0, 3])
def test_varlen_fused_matches_oracle(flags, S):
    """Packed sequences from raw projections: the prologue of the fused forward
    applied per token, then each sequence from its own state."""
    from oracle import prologue as opro
    lengths = [120, 0, 33, 257, 1]
    wl = syn.WORKLOADS["small_layer"].with_(seed=606)
    raw = syn.packed_inputs(wl, lengths, H=2, raw=True)
    q, k, v, beta, d_t = opro.apply(*(f64(raw[n])[None] for n in ("q", "k", "v", "beta_raw", "d_raw")),
                                    b_scale=f64(raw["b_scale"]), qk_norm=flags["qk_norm"])
    ref = ovl.forward(q[0], k[0], v[0], beta[0], d_t[0], f64(raw["A"]), f64(raw["I_prior"]),
                      raw["cu_seqlens"].tolist(), v_star=flags["v_star"])
    g = {n: t.to(DEV) for n, t in raw.items()}
    pal.palimpsa_set_forward_segments(S)
    try:
        out = pal.palimpsa_forward_varlen_fused(g["q"], g["k"], g["v"], g["beta_raw"], g["d_raw"], g["A"],
                                                g["I_prior"], g["cu_seqlens"], g["b_scale"], **flags)
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert pal.palimpsa_get_device_status() == 0
    _check(out, ref)


# ---------------------------------------------------------------- packed training pair

GRAD_PAIRS = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t"), ("dA", "A"),
              ("dI_prior", "I_prior")]


def _bwd_inputs(lengths, H, dk, dv, bf16, with_state, with_final, seed):
    inp = _inputs(lengths, H, dk, dv, bf16, seed)
    N, total = len(lengths), inp["q"].shape[1]
    g = torch.Generator().manual_seed(seed + 1)
    mu0 = torch.randn((N, H, dv, dk), generator=g) if with_state else None
    I0 = (0.5 + 2.0 * torch.rand((N, H, dv, dk), generator=g)) if with_state else None
    dy = torch.randn((H, total, dv), generator=g)
    dmu = torch.randn((N, H, dv, dk), generator=g) if with_final else None
    dI = torch.randn((N, H, dv, dk), generator=g) if with_final else None
    return inp, mu0, I0, dy, dmu, dI


def _bwd_oracle(inp, mu0, I0, dy, dmu, dI):
    f = lambda t: None if t is None else f64(t)
    x = {n: f64(inp[n]) for n in ("q", "k", "v", "beta", "d_t", "A", "I_prior")}
    x.update(mu0=f(mu0), I0=f(I0))
    return ovl.gradients(x, inp["cu_seqlens"].tolist(), f64(dy), f(dmu), f(dI))


def _bwd_gpu(inp, mu0, I0, dy, dmu, dI, checkpointed):
    d = lambda t: None if t is None else t.to(DEV)
    g = {n: t.to(DEV) for n, t in inp.items()}
    ck = None
    if checkpointed:
        _, _, _, ck = pal.palimpsa_forward_varlen_checkpointed(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"],
                                                               g["I_prior"], g["cu_seqlens"], d(mu0), d(I0))
    out = pal.palimpsa_backward_varlen(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"], g["I_prior"],
                                       g["cu_seqlens"], d(mu0), d(I0), d(dy), d(dmu), d(dI), ckpt=ck)
    assert pal.palimpsa_get_device_status() == 0
    return out


BWD_CASES = [
    # (lengths, H, d_k, d_v, bf16, with_state, with_final, checkpointed)
    ([1], 2, 128, 64, True, False, False, False),
    ([5, 0, 17, 1, 64], 3, 128, 64, True, True, True, False),
    ([5, 0, 17, 1, 64], 3, 128, 64, True, True, True, True),
    ([130, 7, 0, 0, 61], 2, 64, 40, False, False, True, True),
    ([33, 96, 2], 1, 64, 128, False, True, False, False),
    ([200, 31, 32, 33], 2, 128, 256, True, True, True, True),
]


@pytest.mark.parametrize("lengths,H,dk,dv,bf16,with_state,with_final,ckpt", BWD_CASES)
def test_varlen_backward_matches_fp64_autograd(lengths, H, dk, dv, bf16, with_state, with_final, ckpt):
    """Gradients through the packed forward: each sequence's own gradients, dA and
    dI_prior summed over sequences, zero rows outside every sequence."""
    case = _bwd_inputs(lengths, H, dk, dv, bf16, with_state, with_final, seed=7000 + sum(lengths) + dv)
    ref = _bwd_oracle(*case)
    out = _bwd_gpu(*case, checkpointed=ckpt)
    pairs = GRAD_PAIRS + ([("dmu0", "mu0"), ("dI0", "I0")] if with_state else [])
    errs = {n: rel_l2(out[n].cpu().numpy(), ref[m]) for n, m in pairs}
    assert max(errs.values()) <= TIGHT, errs


def test_varlen_backward_with_and_without_checkpoints_agree():
    case = _bwd_inputs([300, 45, 1, 199], 2, 128, 64, True, True, True, seed=7101)
    a = _bwd_gpu(*case, checkpointed=False)
    b = _bwd_gpu(*case, checkpointed=True)
    same = {n: rel_l2(a[n].cpu().numpy(), b[n].cpu().numpy()) for n in a}
    assert max(same.values()) <= 1e-5, same


def test_varlen_backward_equal_lengths_equal_the_dense_backward():
    """N equal sequences: the packed kernel does the dense kernel's arithmetic. The
    outputs written without atomics are bit-identical; the atomically summed ones
    (dq, dk, dd_t, dA, dI_prior) agree to rounding order."""
    N, H, T, dk, dv = 3, 2, 150, 128, 64
    inp, mu0, I0, dy, dmu, dI = _bwd_inputs([T] * N, H, dk, dv, True, True, True, seed=7202)
    packed = _bwd_gpu(inp, mu0, I0, dy, dmu, dI, checkpointed=False)
    dense = lambda x: x.reshape((H, N, T) + x.shape[2:]).transpose(0, 1).contiguous()
    g = {n: dense(inp[n]).to(DEV) for n in ("q", "k", "v", "beta", "d_t")}
    ref = pal.palimpsa_backward(g["q"], g["k"], g["v"], g["beta"], g["d_t"], inp["A"].to(DEV), inp["I_prior"].to(DEV),
                                mu0.to(DEV), I0.to(DEV), dense(dy).to(DEV), dmu.to(DEV), dI.to(DEV))
    for n in ("dv", "dbeta"):
        assert torch.equal(dense(packed[n].cpu()), ref[n].cpu()), n
    for n in ("dmu0", "dI0"):
        assert torch.equal(packed[n], ref[n]), n
    for n in ("dq", "dk", "dd_t"):
        assert rel_l2(dense(packed[n].cpu()).numpy(), ref[n].cpu().numpy()) <= 1e-6, n
    for n in ("dA", "dI_prior"):
        assert rel_l2(packed[n].cpu().numpy(), ref[n].cpu().numpy()) <= 1e-6, n


def test_varlen_backward_bad_offsets_are_reported_not_faulted():
    """Offsets that break the rules: that sequence's CTAs touch nothing, the call
    latches a domain error, the other sequences' gradients are still right."""
    lengths = [20, 30, 10]
    inp, mu0, I0, dy, dmu, dI = _bwd_inputs(lengths, 2, 128, 64, True, True, True, seed=7303)
    ref = _bwd_oracle(inp, mu0, I0, dy, dmu, dI)
    g = {n: t.to(DEV) for n, t in inp.items()}
    d = lambda t: t.to(DEV)
    for cu in ([0, 20, 15, 60], [0, 20, 50, 60 + 40], [0, 20, 50, 60]):
        cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
        out = pal.palimpsa_backward_varlen(g["q"], g["k"], g["v"], g["beta"], g["d_t"], g["A"], g["I_prior"], cu_d,
                                           d(mu0), d(I0), d(dy), d(dmu), d(dI), max_seqlen=25)
        assert pal.palimpsa_get_device_status() == 5  # PALIMPSA_ERR_DOMAIN
        for n, m in (("dq", "q"), ("dv", "v"), ("dd_t", "d_t")):
            assert rel_l2(out[n][:, :20].cpu().numpy(), ref[m][:, :20]) <= TIGHT, n
        assert rel_l2(out["dmu0"][0].cpu().numpy(), ref["mu0"][0]) <= TIGHT
    out = _bwd_gpu(inp, mu0, I0, dy, dmu, dI, checkpointed=False)
    errs = {n: rel_l2(out[n].cpu().numpy(), ref[m]) for n, m in GRAD_PAIRS}
    assert max(errs.values()) <= TIGHT, errs


def test_varlen_checkpoints_are_each_sequences_states():
    """Checkpoint c of sequence n (from token s0) sits in slot s0 // 32 + n + c
    of each head and holds its state before its token 32 c, as (M = I mu, I)
    per value row, from the forward split into segments or not."""
    lengths = [70, 0, 33, 5]
    inp = _inputs(lengths, 2, 128, 64, True, seed=7404)
    cu = inp["cu_seqlens"].tolist()
    g = {n: t.to(DEV) for n, t in inp.items()}
    for S in (0, 2):
        pal.palimpsa_set_forward_segments(S)
        try:
            _, _, _, ck = pal.palimpsa_forward_varlen_checkpointed(g["q"], g["k"], g["v"], g["beta"], g["d_t"],
                                                                   g["A"], g["I_prior"], g["cu_seqlens"])
        finally:
            pal.palimpsa_set_forward_segments(0)
        assert pal.palimpsa_get_device_status() == 0
        ck = ck.cpu().numpy()
        for n, L in enumerate(lengths):
            for c in range(-(-L // 32)):
                t = 32 * c
                sub = {m: inp[m][:, cu[n]:cu[n] + t] for m in ("q", "k", "v", "beta", "d_t")}
                sub["cu_seqlens"] = torch.tensor([0, t], dtype=torch.int32)
                sub.update(A=inp["A"], I_prior=inp["I_prior"])
                _, mu_r, I_r = _oracle(sub)
                slot = cu[n] // 32 + n + c
                assert rel_l2(ck[:, slot, :, 0, :], mu_r[0] * I_r[0]) <= TIGHT, (n, c)
                assert rel_l2(ck[:, slot, :, 1, :], I_r[0]) <= TIGHT, (n, c)


def test_varlen_backward_bench_packing_sampled_sequences():
    """The packed training pair at the benchmark's packing of the small layer (its
    B*T tokens per head as 4*B ragged sequences, bf16): the checkpointed forward
    and the backward reading its checkpoints, against fp64 autograd on two
    sequences of one head."""
    from oracle import autograd as ag
    wl = syn.WORKLOADS["small_layer"]
    lengths = syn.varlen_lengths(wl.B * wl.T, 4 * wl.B, wl.seed)
    pk = syn.packed_inputs(wl, lengths, H=wl.H, seed=wl.seed)
    g = torch.Generator().manual_seed(77)
    dy = torch.randn((wl.H, wl.B * wl.T, wl.d_v), generator=g)
    d = {n: t.to(DEV) for n, t in pk.items()}
    _, _, _, ck = pal.palimpsa_forward_varlen_checkpointed(d["q"], d["k"], d["v"], d["beta"], d["d_t"], d["A"],
                                                           d["I_prior"], d["cu_seqlens"])
    out = pal.palimpsa_backward_varlen(d["q"], d["k"], d["v"], d["beta"], d["d_t"], d["A"], d["I_prior"],
                                       d["cu_seqlens"], None, None, dy.to(DEV), want_state_grads=False, ckpt=ck)
    assert pal.palimpsa_get_device_status() == 0
    cu = pk["cu_seqlens"].tolist()
    h = 3
    f = syn.as_float64_numpy
    for n in (0, int(np.argmax(lengths))):
        s0, s1 = cu[n], cu[n + 1]
        sub = {m: f(pk[m][h:h + 1, s0:s1])[None] for m in ("q", "k", "v", "beta", "d_t")}
        sub.update(A=f(pk["A"][h:h + 1]), I_prior=f(pk["I_prior"][h:h + 1]), mu0=None, I0=None)
        ref = ag.gradients(sub, f(dy[h:h + 1, s0:s1])[None])
        for name, m in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dd_t", "d_t")):
            assert rel_l2(out[name][h:h + 1, s0:s1].cpu().numpy(), ref[m][0]) <= TIGHT, (n, name)
