"""Seeded synthetic inputs shaped like the language-model layers the Palimpsa
pages describe. This module only draws random numbers: it holds none of the
recurrence's arithmetic, and both the CUDA path and the fp64 oracle consume
exactly what it returns (bf16 inputs are rounded here, once, and the oracle
upcasts the rounded values exactly).

Recipes (all heads share one recipe; the draws happen in the order
A, key pool, d_t, q, k, v, beta from one torch Generator seeded per workload):

* q, k ~ N(0, 1) then L2-normalised per token (the query/key L2 norm of the
  Palimpsa-D block, slide 10); for ``long_context`` the keys come from a fixed
  pool of 512 unit vectors, each token picking one uniformly and adding
  Gaussian jitter of norm ~0.1 before renormalising (heavy key interference).
* v ~ N(0, 1); beta = sigmoid(N(0, 1)) per value channel (beta >= 0, slide 4).
* d_t = softplus(N(m, s)) per head-token (alpha = exp(-A d_t), slide 5).
* A = 0.5 for ``tiny``, else U(0.1, 1) per head; I_prior = 1 per head;
  mu0 = 0 and I0 = I_prior.

``raw=True`` returns the same draws before any activation, for the fused
prologue: q and k as drawn (pooled keys with their jitter, not renormalised),
beta_raw ~ N(0, 1), d_raw ~ N(m, s), v as drawn (read as v* in the v* mode),
plus a per-head b_scale ~ U(0.1, 1) (slide 11's fine-tuning range) drawn after
everything else, so the other tensors equal the activated recipe's draws.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int            # tokens of the scan (the prefill length for ``decode``)
    d_k: int
    d_v: int
    bf16: bool        # q, k, v, beta in bf16 (state and y are always fp32)
    chunk: int
    dt_mean: float
    dt_std: float
    A_fixed: float | None
    key_pool: int = 0
    key_jitter: float = 0.0
    steps: int = 0    # decode steps after the scan (``decode`` only)
    seed: int = 0

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * (self.T + self.steps)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # 1 x 2 heads x 256 tokens, d_k = d_v = 64, fp32: the case the oracle finishes in seconds.
    "tiny": Workload("tiny", 1, 2, 256, 64, 64, False, 64, 0.0, 1.0, 0.5, seed=20260),
    # 4 x 16 heads x 2048 tokens, d_k = 128, d_v = 64, bf16 inputs.
    "small_layer": Workload("small_layer", 4, 16, 2048, 128, 64, True, 64, 0.0, 1.0, None, seed=20261),
    # 8 x 24 heads x 4096 tokens (a 760M-scale layer), windows from a few to thousands of tokens.
    "layer_760m": Workload("layer_760m", 8, 24, 4096, 128, 64, True, 64, -1.0, 1.0, None, seed=20262),
    # 1 x 32 heads x 32768 tokens with pooled, jittered keys and long memory.
    "long_context": Workload("long_context", 1, 32, 32768, 128, 64, True, 64, -2.0, 0.5, None,
                             key_pool=512, key_jitter=0.1, seed=20263),
    # 256 x 32 heads: a 512-token prefill with layer_760m statistics, then 1024 decode steps.
    "decode": Workload("decode", 256, 32, 512, 128, 64, True, 64, -1.0, 1.0, None, steps=1024, seed=20264),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _unit(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def _draw(wl: Workload, lead: tuple, H: int, g, device, pool=None, raw=False):
    """Draw q, k, v, beta, d_t with leading shape `lead` (ending in H); with
    `raw`, the pre-activation values (q, k, v, beta_raw, d_raw)."""
    dk, dv = wl.d_k, wl.d_v
    f32 = torch.float32
    act = (lambda f, x: x) if raw else (lambda f, x: f(x))
    d_t = act(F.softplus, wl.dt_mean + wl.dt_std * torch.randn(lead, generator=g, device=device, dtype=f32))
    q = act(_unit, torch.randn(lead + (dk,), generator=g, device=device, dtype=f32))
    if wl.key_pool:
        idx = torch.randint(0, wl.key_pool, lead, generator=g, device=device)
        eps = torch.randn(lead + (dk,), generator=g, device=device, dtype=f32) * (wl.key_jitter / dk ** 0.5)
        k = act(_unit, pool[idx] + eps)
    else:
        k = act(_unit, torch.randn(lead + (dk,), generator=g, device=device, dtype=f32))
    v = torch.randn(lead + (dv,), generator=g, device=device, dtype=f32)
    beta = act(torch.sigmoid, torch.randn(lead + (dv,), generator=g, device=device, dtype=f32))
    if wl.bf16:
        q, k, v, beta = (x.to(torch.bfloat16) for x in (q, k, v, beta))
    return q, k, v, beta, d_t


def sequence_inputs(wl: Workload, *, B=None, H=None, T=None, device="cpu", seed=None, raw=False):
    """Inputs of one scan: q, k [B,H,T,d_k]; v, beta [B,H,T,d_v]; d_t [B,H,T];
    A, I_prior [H]. Returns a dict of contiguous tensors on `device`. With
    `raw`, the keys are q, k, v, beta_raw, d_raw, A, I_prior, b_scale."""
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    T = wl.T if T is None else T
    g = _gen(device, wl.seed if seed is None else seed)
    f32 = torch.float32
    if wl.A_fixed is not None:
        A = torch.full((H,), wl.A_fixed, dtype=f32, device=device)
    else:
        A = 0.1 + 0.9 * torch.rand((H,), generator=g, device=device, dtype=f32)
    pool = None
    if wl.key_pool:
        pool = _unit(torch.randn((wl.key_pool, wl.d_k), generator=g, device=device, dtype=f32))
    q, k, v, beta, d_t = _draw(wl, (B, H, T), H, g, device, pool, raw)
    I_prior = torch.ones((H,), dtype=f32, device=device)
    if raw:
        b_scale = 0.1 + 0.9 * torch.rand((H,), generator=g, device=device, dtype=f32)
        return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(), "beta_raw": beta.contiguous(),
                "d_raw": d_t.contiguous(), "A": A, "I_prior": I_prior, "b_scale": b_scale}
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(), "beta": beta.contiguous(),
            "d_t": d_t.contiguous(), "A": A, "I_prior": I_prior}


def decode_inputs(wl: Workload, steps: int, *, B=None, H=None, device="cpu", seed=None, raw=False):
    """Per-step decode inputs stacked over steps: q, k [S,B,H,d_k]; v, beta
    [S,B,H,d_v]; d_t [S,B,H] (the same statistics as the scan). A and I_prior
    are those of the prefill (same seed), so pass ``sequence_inputs``' A.
    With `raw`: q, k, v, beta_raw, d_raw before activation."""
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    g = _gen(device, (wl.seed if seed is None else seed) * 7919 + 1)
    q, k, v, beta, d_t = _draw(wl, (steps, B, H), H, g, device, raw=raw)
    names = ("beta_raw", "d_raw") if raw else ("beta", "d_t")
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(), names[0]: beta.contiguous(),
            names[1]: d_t.contiguous()}


def as_float64_numpy(t: torch.Tensor):
    """Exact upcast of (possibly bf16-rounded) inputs for the fp64 oracle."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def varlen_lengths(total: int, n: int, seed: int):
    """n sequence lengths summing to `total`: a seeded uniform mix, each at least 1
    (requires n <= total). Only draws numbers; the packing is the caller's."""
    g = torch.Generator().manual_seed(int(seed))
    w = 0.05 + torch.rand((n,), generator=g, dtype=torch.float64)
    raw = (w / w.sum() * (total - n)).floor().to(torch.int64) + 1
    raw[-1] += total - int(raw.sum())
    return [int(x) for x in raw]


def packed_inputs(wl: Workload, lengths, *, H=None, device="cpu", seed=None, raw=False):
    """A packed variable-length batch with the workload's recipe: q, k
    [H, total_T, d_k]; v, beta [H, total_T, d_v]; d_t [H, total_T]; A, I_prior
    [H]; cu_seqlens [N + 1] int32 with sequence n = tokens [cu[n], cu[n+1]).
    With `raw`, the pre-activation draws as in ``sequence_inputs``."""
    H = wl.H if H is None else H
    total = int(sum(lengths))
    inp = sequence_inputs(wl, B=1, H=H, T=total, device=device, seed=seed, raw=raw)
    out = {k: (v[0].contiguous() if v.dim() >= 3 else v) for k, v in inp.items()}
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device=device)
    return out
