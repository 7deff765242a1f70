"""The library's scratch memory: what it keeps between calls and what it gives back.

The time-split forward and the backward take device scratch for the length of
one call from a stream-ordered pool the library owns. Freed pages stay mapped
for the next call up to a retention bound (512 MiB by default), so that the
forward does not pay to map fresh pages each call; at a synchronisation the
pool gives back whatever it holds above the bound, and palimpsa_release_scratch
gives back everything. These tests read the pool's mapped bytes through the C
ABI around forwards and backwards of known scratch sizes."""
import pytest
import torch

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
DEV = "cuda"
MiB = 1 << 20
DEFAULT_RETENTION = 512 * MiB


def _fwd(gi, **kw):
    out = pal.palimpsa_forward_chunked(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"],
                                       **kw)
    assert pal.palimpsa_get_device_status() == 0
    return out


def _bwd(gi, seed):
    B, H, T, _ = gi["q"].shape
    dv = gi["v"].shape[-1]
    g = torch.Generator(device=DEV).manual_seed(seed)
    dy = torch.randn((B, H, T, dv), generator=g, device=DEV)
    out = pal.palimpsa_backward(gi["q"], gi["k"], gi["v"], gi["beta"], gi["d_t"], gi["A"], gi["I_prior"], None, None,
                                dy, want_state_grads=False)
    assert pal.palimpsa_get_device_status() == 0
    return out


def test_scratch_is_kept_up_to_the_bound_and_released_on_request():
    pal.palimpsa_set_scratch_retention(DEFAULT_RETENTION)
    pal.palimpsa_release_scratch()
    assert pal.palimpsa_scratch_reserved_bytes() == 0

    # a time-split forward: its scratch (a few MiB) is below the bound and stays mapped
    wl = syn.WORKLOADS["small_layer"].with_(B=1, H=4, T=1024)
    gi = {k: v.to(DEV) for k, v in syn.sequence_inputs(wl, seed=71).items()}
    pal.palimpsa_set_forward_segments(6)
    try:
        plan = pal.palimpsa_forward_plan(wl.B, wl.H, wl.T, wl.d_k, wl.d_v, chunk=wl.chunk, bf16=wl.bf16)
        assert plan["segments"] > 1 and plan["scratch_bytes"] > 0
        first = _fwd(gi, chunk=wl.chunk)
        torch.cuda.synchronize()
        kept = pal.palimpsa_scratch_reserved_bytes()
        assert kept >= plan["scratch_bytes"]

        # a backward whose scratch (B*H*d_v/8 CTAs x ceil(T/32) x 8 KiB = 600 MiB) is above the
        # bound: once the device synchronises, the pool holds no more than the bound
        big = syn.WORKLOADS["small_layer"].with_(B=4, H=16, T=4800)
        gb = {k: v.to(DEV) for k, v in syn.sequence_inputs(big, seed=72).items()}
        need = 4 * 16 * (64 // 8) * (-(-4800 // 32)) * 8 * 128 * 2 * 4
        assert need > DEFAULT_RETENTION
        _bwd(gb, 73)
        torch.cuda.synchronize()
        assert pal.palimpsa_scratch_reserved_bytes() <= DEFAULT_RETENTION

        # with a larger bound the same backward's scratch stays mapped ...
        pal.palimpsa_set_scratch_retention(4 << 30)
        _bwd(gb, 73)
        torch.cuda.synchronize()
        assert pal.palimpsa_scratch_reserved_bytes() >= need
        # ... until the caller asks for it back
        pal.palimpsa_release_scratch()
        assert pal.palimpsa_scratch_reserved_bytes() == 0

        # the pool serves the next call as before, with the same results
        again = _fwd(gi, chunk=wl.chunk)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    finally:
        pal.palimpsa_set_forward_segments(0)
        pal.palimpsa_set_scratch_retention(DEFAULT_RETENTION)


def test_zero_retention_keeps_nothing_after_a_synchronisation():
    pal.palimpsa_set_scratch_retention(0)
    try:
        wl = syn.WORKLOADS["small_layer"].with_(B=1, H=2, T=700)
        gi = {k: v.to(DEV) for k, v in syn.sequence_inputs(wl, seed=74).items()}
        _bwd(gi, 75)
        torch.cuda.synchronize()
        assert pal.palimpsa_scratch_reserved_bytes() == 0
    finally:
        pal.palimpsa_set_scratch_retention(DEFAULT_RETENTION)
