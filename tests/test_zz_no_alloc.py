"""The forward entry point that allocates nothing (palimpsa_forward_chunked_noalloc).

Some callers cannot let a library allocate device memory: a serving process
that reserves all of it at start-up, a plugin inside a framework that owns the
device heap, a latency-critical loop. For them the time-split scratch of the
chunked forward lives in a fixed array inside the library. These tests call
that entry point through the C ABI and compare it with the allocating entry
point on the same inputs, twice in a row (the array keeps the previous call's
contents, which must not leak into the next result) and with the fp64 oracle,
so that a fault shared by both entry points (the time-split code they have in
common) cannot pass unseen; and check that a call needing more scratch than the
array holds is refused without touching its outputs. This file is collected
last on purpose.
"""
import ctypes

import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import synthetic as syn
from tests._helpers import TIGHT, oracle_forward_from, rel_l2, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"
ERR_SCRATCH_LIMIT = 9
NOALLOC_SCRATCH_BYTES = 16 << 20     # the fixed array's size, as the header states


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(fn, gi, mu0, I0, y, mu_T, I_T, chunk):
    B, H, T, dk = gi["q"].shape
    dv = gi["v"].shape[-1]
    dtype = 1 if gi["q"].dtype == torch.bfloat16 else 0
    return fn(_ptr(gi["q"]), _ptr(gi["k"]), _ptr(gi["v"]), _ptr(gi["beta"]), _ptr(gi["d_t"]), _ptr(gi["A"]),
              _ptr(gi["I_prior"]), _ptr(mu0), _ptr(I0), _ptr(y), _ptr(mu_T), _ptr(I_T), B, H, T, dk, dv, chunk,
              dtype, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_both(lib, wl, seed, with_state):
    inp = syn.sequence_inputs(wl, seed=seed)
    gi = {k: v.to(DEV) for k, v in inp.items()}
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.d_k, wl.d_v
    mu0 = I0 = None
    if with_state:
        g = torch.Generator().manual_seed(seed + 1)
        mu0 = torch.randn((B, H, dv, dk), generator=g).to(DEV)
        I0 = (0.5 + 3.0 * torch.rand((B, H, dv, dk), generator=g)).to(DEV)
    outs = []
    for fn in (lib.palimpsa_forward_chunked, lib.palimpsa_forward_chunked_noalloc):
        y = torch.full((B, H, T, dv), float("nan"), device=DEV)
        mu_T = torch.full((B, H, dv, dk), float("nan"), device=DEV)
        I_T = torch.full((B, H, dv, dk), float("nan"), device=DEV)
        assert _call(fn, gi, mu0, I0, y, mu_T, I_T, wl.chunk) == 0
        assert pal.palimpsa_get_device_status() == 0
        outs.append((y, mu_T, I_T))
    for ref, got in zip(outs[0], outs[1]):
        assert torch.isfinite(got).all()
        assert rel_l2(got.cpu(), ref.cpu()) <= min(tol_for(inp), TIGHT)
    # the no-allocation results against the oracle on the same inputs, every head
    oref = oracle_forward_from(inp, None if mu0 is None else mu0.cpu(), None if I0 is None else I0.cpu())
    for got, ref in zip(outs[1], oref):
        assert rel_l2(got.cpu().numpy(), ref) <= min(tol_for(inp), TIGHT)


def _assert_split_fits(wl):
    """The plan of this call splits time (so the fixed array is used) and fits the array."""
    plan = pal.palimpsa_forward_plan(wl.B, wl.H, wl.T, wl.d_k, wl.d_v, chunk=wl.chunk, bf16=wl.bf16)
    assert plan["segments"] > 1, plan
    assert 0 < plan["scratch_bytes"] <= NOALLOC_SCRATCH_BYTES, plan


def test_no_alloc_forward_matches_the_allocating_one_twice_in_a_row():
    lib = pal.load_library()
    pal.palimpsa_set_forward_segments(0)
    try:
        # call 1: few heads, so the automatic plan splits time and uses the scratch array
        wl1 = syn.WORKLOADS["small_layer"].with_(B=1, H=4, T=600)
        _assert_split_fits(wl1)
        _run_both(lib, wl1, seed=501, with_state=True)
        # call 2: another shape and a forced split, over what call 1 left in the array
        pal.palimpsa_set_forward_segments(5)
        wl2 = syn.WORKLOADS["small_layer"].with_(B=2, H=3, T=333, d_k=64, d_v=24, bf16=False, chunk=32)
        _assert_split_fits(wl2)
        _run_both(lib, wl2, seed=502, with_state=False)
    finally:
        pal.palimpsa_set_forward_segments(0)


def test_no_alloc_forward_refuses_calls_beyond_its_scratch():
    lib = pal.load_library()
    wl = syn.WORKLOADS["small_layer"].with_(B=4, H=32, T=256)   # 128 heads x 7 boundaries x 64 KiB > 16 MiB
    inp = syn.sequence_inputs(wl, seed=503)
    gi = {k: v.to(DEV) for k, v in inp.items()}
    y = torch.full((4, 32, 256, 64), 7.0, device=DEV)
    mu_T = torch.full((4, 32, 64, 128), 7.0, device=DEV)
    I_T = torch.full((4, 32, 64, 128), 7.0, device=DEV)
    pal.palimpsa_set_forward_segments(8)
    try:
        rc = _call(lib.palimpsa_forward_chunked_noalloc, gi, None, None, y, mu_T, I_T, 32)
    finally:
        pal.palimpsa_set_forward_segments(0)
    assert rc == ERR_SCRATCH_LIMIT
    assert "scratch" in pal.palimpsa_status_string(rc)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()) and bool((mu_T == 7.0).all()) and bool((I_T == 7.0).all())
    assert pal.palimpsa_get_device_status() == 0
