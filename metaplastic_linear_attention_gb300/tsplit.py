"""Time-sharded forward: the T tokens of the same B x H sequences split into
consecutive shards over the ranks of a process group (rank order = time
order), with one exchange.

Source: Bonnet et al., "Learning to Remember, Learn, and Forget in
Attention-Based Models" — slide 9 (App. A.12): in the natural parameters
M = I (.) mu and Ibar = I - I_prior both recurrences are affine in the state
with the shared scalar decay alpha, so each shard acts on the state as
(M, Ibar) -> Gamma (M, Ibar) + (dM, dIbar). Rank r

1. computes its shard's (dM, dIbar, Gamma) from a zero state
   (``palimpsa_segment_summary``),
2. all-gathers every rank's summary (the one exchange: 8 d_v d_k + 4 bytes per
   head and rank),
3. folds the summaries of ranks 0 .. r-1 into the initial state
   (``palimpsa_state_combine``), and
4. runs the forward on its own tokens from that state.

Every step of the arithmetic runs in the library's kernels. This module only
moves tensors and calls the collective. The operations are passed in as a
``ShardOps`` so that the exchange can be exercised on CPU ranks with other
implementations of the three steps. The library itself has no CPU path.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch
import torch.distributed as dist

from . import binding


@dataclass(frozen=True)
class ShardOps:
    # (q, k, v, beta, d_t, A, I_prior) -> (summary [B,H,2,d_v,d_k], gamma [B,H])
    summary: Callable
    # (summaries [R,B,H,2,d_v,d_k], gammas [R,B,H], I_prior, mu0, I0) -> (mu, I) [B,H,d_v,d_k]
    combine: Callable
    # (q, k, v, beta, d_t, A, I_prior, mu0, I0) -> (y, mu_T, I_T)
    forward: Callable


def library_ops(chunk: int = 0, stream=None) -> ShardOps:
    """The three steps as calls into the CUDA library."""
    return ShardOps(
        summary=lambda q, k, v, beta, d_t, A, Ip: binding.palimpsa_segment_summary(
            q, k, v, beta, d_t, A, Ip, chunk=chunk, stream=stream),
        combine=lambda S, G, Ip, mu0, I0: binding.palimpsa_state_combine(S, G, Ip, mu0, I0, stream=stream),
        forward=lambda q, k, v, beta, d_t, A, Ip, mu0, I0: binding.palimpsa_forward_chunked(
            q, k, v, beta, d_t, A, Ip, mu0, I0, chunk=chunk, stream=stream),
    )


def forward_time_sharded(q, k, v, beta, d_t, A, I_prior, mu0=None, I0=None, *, group=None, ops: ShardOps = None):
    """This rank's shard of the forward: q, k [B,H,T_r,d_k], v, beta
    [B,H,T_r,d_v], d_t [B,H,T_r] are the rank's consecutive tokens; A, I_prior,
    mu0, I0 are the same on every rank. Returns (y of the shard, state at the
    end of the shard); on the last rank that state is the sequences' final state.
    Shards may have different lengths, including zero."""
    ops = ops or library_ops()
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    summ, gam = ops.summary(q, k, v, beta, d_t, A, I_prior)
    n = summ.numel()
    flat = torch.cat([summ.reshape(-1), gam.reshape(-1)])
    parts = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(parts, flat, group=group)
    before = parts[:rank]
    if before:
        S = torch.stack([p[:n].view(summ.shape) for p in before])
        G = torch.stack([p[n:].view(gam.shape) for p in before])
    else:
        S = summ.new_empty((0,) + tuple(summ.shape))
        G = gam.new_empty((0,) + tuple(gam.shape))
    mu_s, I_s = ops.combine(S, G, I_prior, mu0, I0)
    return ops.forward(q, k, v, beta, d_t, A, I_prior, mu_s, I_s)
