#!/usr/bin/env python3
"""Benchmark of the Palimpsa dual-state recurrence on GB300.

Default workload ("decode"): B=256, H=32, d_k=128, d_v=64, bf16 inputs, fp32
state. One step = the whole job: a 512-token chunked prefill (forward_chunked)
that leaves mu, I resident in HBM, then 1024 recurrent decode steps
(palimpsa_step) on that state. The metric is head-tokens processed per second
(B*H*(512 + 1024) per step); the dominant kernel is the decode step, bound by
HBM bandwidth (it streams the 537 MB state in and out every token).

Other workloads (``--workload small_layer|layer_760m|long_context|tiny``): one
step = one chunked forward over the whole configuration (ALU-bound).

Prints ONE JSON line on rank 0. ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Palimpsa scan throughput (B·H·T tokens/s) and % of GB300 HBM roofline"
UNIT = "head-tokens/s"
FALLBACK_HBM_GBS = 6800.0
# The ALU-bound kernels (chunked forward, backward) spend one SFU reciprocal per
# element-token; their roofline is the reciprocal rate per clock and SM, measured
# live by the library's issue-rate probe, x the SM count x the maximum SM clock.
# The backward is also set against the FP32 arithmetic it cannot avoid, per
# element-token: one forward step to recover the state (I and M: two FMA each),
# mu = M r, the adjoint step (q r, dy q r, its product with mu, and the two carried
# FMAs of gM and gI) and the gradient sums (dq: 1, dk: 2, the two row sums, and J:
# 1), 16 operations at the probe's FP32 FMA rate.
BWD_MIN_FP32_OPS = 16

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel from one ncu
# capture, valid only while the kernel's source file is byte-identical to the one captured
# (sha256 below); otherwise null. The decode step's figure is the mean of four consecutive
# steady-state steps at the full B=256, H=32 state (a 64-token prefill and 16 decode tokens
# per bench step keep the device footprint near 1 GB), captured without cache flushes
# (--cache-control none) as they run in the timed region: each step finds the rows the
# previous one stored last still in L2. The traffic of a step does not depend on the prefill's
# length or the number of steps after the first.
NCU_TRAFFIC = {
    "palimpsa_step": {"bytes_per_launch": 932406848, "source": "csrc/step.cu",
                      "sha256": "a99e48cc88dad37e653c648b985da9e595766bb149603d3a12dfc0fe1c5e09b3"},
}


def _captured_traffic(kernel):
    import hashlib
    rec = NCU_TRAFFIC.get(kernel)
    if rec is None:
        return None
    path = os.path.join(ROOT, "metaplastic_linear_attention_gb300", rec["source"])
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec["bytes_per_launch"] if digest == rec["sha256"] else None


# ----------------------------------------------------------------------------- helpers

def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = os.path.join("/tmp", f"palimpsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.out) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        try:
            os.remove(self.out)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- multi-rank host logic

def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_bootstrap(rank, n, port, target, args):
    """Entry of one spawned rank: the environment torchrun would give it, then the target."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(n), LOCAL_WORLD_SIZE=str(n),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    target(*args)


def spawn_ranks(n: int, target, args=(), poll_s: float = 0.2):
    """Run target(*args) as n local ranks, one process each (rank r on GPU r), with
    RANK, LOCAL_RANK, WORLD_SIZE and MASTER_ADDR/MASTER_PORT (127.0.0.1, a free port)
    set as torchrun sets them. Processes start with the spawn method, so none
    inherits a CUDA context. Waits for all of them; if one fails, the others are
    stopped (they could otherwise wait forever at a barrier) and SystemExit is
    raised naming the failed ranks."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_bootstrap, args=(r, n, port, target, tuple(args))) for r in range(n)]
    for pr in procs:
        pr.start()
    failed = []
    while True:
        alive = [pr for pr in procs if pr.exitcode is None]
        failed = [r for r, pr in enumerate(procs) if pr.exitcode not in (None, 0)]
        if failed or not alive:
            break
        alive[0].join(poll_s)
    if failed:
        for pr in procs:
            if pr.exitcode is None:
                pr.terminate()
        for pr in procs:
            pr.join()
        raise SystemExit(f"bench: rank(s) {failed} of {n} failed "
                         f"(exit codes {[procs[r].exitcode for r in failed]})")


def _run_rank(argv):
    main(argv)


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank runs an independent replica of the workload (weak scaling): its own inputs."""
    return base_seed + 1000 * rank


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The slowest rank's value (timings are taken as the max over ranks)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ws: int, seconds: float) -> float:
    """Units processed by all ranks together per second of the slowest rank."""
    return units_per_rank * ws / seconds


# ----------------------------------------------------------------------------- byte / work accounting

def decode_step_bytes(B, H, dk, dv, in_bytes):
    """Algorithmic HBM bytes of one palimpsa_step launch: mu and I read and written
    (16 B per state element) plus q, k, v, beta, d_t in and y out."""
    state = B * H * dv * dk * 4 * 2 * 2
    inputs = B * H * (2 * dk + 2 * dv) * in_bytes + B * H * 4 + 2 * H * 4
    out = B * H * dv * 4
    return state + inputs + out


def forward_bytes(B, H, T, dk, dv, in_bytes):
    """Algorithmic HBM bytes of one forward_chunked launch: every input once, y
    once, the final state written once (the initial state is synthesised)."""
    per_tok = (2 * dk + 2 * dv) * in_bytes + 4 + dv * 4
    return B * H * T * per_tok + B * H * dv * dk * 4 * 2 + 2 * H * 4


# ----------------------------------------------------------------------------- our implementation

def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    import metaplastic_linear_attention_gb300 as pal
    from metaplastic_linear_attention_gb300 import build_lib
    from metaplastic_linear_attention_gb300 import synthetic as syn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    build_lib.build()
    pal.load_library()
    rates = issue_rates(pal)
    wl = _workload(args)
    seed = replica_seed(wl.seed, rank)
    inp = syn.sequence_inputs(wl, device=dev, seed=seed)
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.d_k, wl.d_v
    in_bytes = 2 if wl.bf16 else 4
    S = wl.steps
    dec = syn.decode_inputs(wl, S, device=dev, seed=seed) if S else None
    f32 = torch.float32
    y_pre = torch.empty((B, H, T, dv), dtype=f32, device=dev)
    mu = torch.empty((B, H, dv, dk), dtype=f32, device=dev)
    I = torch.empty((B, H, dv, dk), dtype=f32, device=dev)
    y_dec = torch.empty((max(S, 1), B, H, dv), dtype=f32, device=dev)
    stream = torch.cuda.current_stream()

    ev = []

    def one_step(record=False):
        e0 = torch.cuda.Event(enable_timing=True) if record else None
        e1 = torch.cuda.Event(enable_timing=True) if record else None
        e2 = torch.cuda.Event(enable_timing=True) if record else None
        if record:
            e0.record(stream)
        pal.palimpsa_forward_chunked(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"],
                                     inp["I_prior"], y=y_pre, mu_T=mu, I_T=I, chunk=wl.chunk)
        if record:
            e1.record(stream)
        if S:  # the S tokens in order, one palimpsa_step launch each
            pal.palimpsa_step(dec["q"], dec["k"], dec["v"], dec["beta"], dec["d_t"], inp["A"], inp["I_prior"], mu, I,
                              y=y_dec[:S])
        if record:
            e2.record(stream)
            ev.append((e0, e1, e2))

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    st = pal.palimpsa_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {pal.palimpsa_status_string(st)}")

    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for _ in range(args.steps):
            one_step(record=True)
        t_end.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    pre_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    ms_total = max_over_ranks(ms_total, ws, dev)
    clocks = clk.summary()
    st = pal.palimpsa_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {pal.palimpsa_status_string(st)}")

    ms_step = ms_total / args.steps
    # kernel launches of one forward call: 1, or 3 when the planner splits time
    fwd_launches = pal.palimpsa_forward_plan(B, H, T, dk, dv, chunk=wl.chunk, bf16=wl.bf16)["launches"]
    head_tokens = B * H * (T + S)
    value = whole_job_rate(head_tokens, ws, ms_step / 1e3)

    peaks, peak_kind = _measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    kernels = {}
    fwd_avg_ms = statistics.mean(pre_ms)
    fb = forward_bytes(B, H, T, dk, dv, in_bytes)
    E_fwd = B * H * T * dv * dk
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rcp_rate = rates["rcp"]
    alu_peak = n_sms * rcp_rate * sm_max * 1e6 / 1e9   # G element-updates/s
    kernels["palimpsa_fwd_chunked"] = {
        "launches_per_step": 1, "avg_ms": fwd_avg_ms,
        "head_tokens_per_s": B * H * T / (fwd_avg_ms / 1e3),
        "hbm_gbs": fb / (fwd_avg_ms / 1e3) / 1e9,
        "alu": {"achieved": E_fwd / (fwd_avg_ms / 1e3) / 1e9, "peak": alu_peak, "unit": "G element-updates/s",
                "frac": E_fwd / (fwd_avg_ms / 1e3) / 1e9 / alu_peak},
    }
    if S:
        dec_avg_ms = statistics.mean(dec_ms) / S
        db = decode_step_bytes(B, H, dk, dv, in_bytes)
        ach = db / (dec_avg_ms / 1e3) / 1e9
        kernels["palimpsa_step"] = {"launches_per_step": S, "avg_ms": dec_avg_ms,
                                    "head_tokens_per_s": B * H / (dec_avg_ms / 1e3), "hbm_gbs": ach,
                                    "bytes_per_launch": db}
        traffic = args.traffic if args.traffic is not None else (
            _captured_traffic("palimpsa_step") if (B, H, dk, dv) == (256, 32, 128, 64) and wl.bf16 else None)
        roofline = {"bound": "hbm", "kernel": "palimpsa_step", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                    "frac": ach / hbm_peak, "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                    "bytes_per_launch": db}
        if traffic:
            # DRAM's own rate over the step: the measured bytes per launch (less than the
            # algorithmic ones, as consecutive steps hand rows over in L2) over the live time
            roofline["dram_gbs"] = traffic / (dec_avg_ms / 1e3) / 1e9
            roofline["dram_frac"] = roofline["dram_gbs"] / hbm_peak
    else:
        a = kernels["palimpsa_fwd_chunked"]["alu"]
        roofline = {"bound": "alu", "kernel": "palimpsa_fwd_chunked", "achieved": a["achieved"], "peak": alu_peak,
                    "unit": "G element-updates/s", "frac": a["frac"], "traffic": args.traffic,
                    "peak_source": f"{n_sms} SMs x {rcp_rate:.2f} rcp/clk/SM (measured by palimpsa_probe_issue_rate) "
                                   f"x {sm_max:.0f} MHz"}

    # The "without Meta" comparator (importance frozen at I_prior) on the same scan
    # inputs, timed outside the timed region: what metaplasticity costs here.
    def _nometa():
        pal.palimpsa_forward_without_meta(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"],
                                          inp["I_prior"], y=y_pre, mu_T=mu, chunk=wl.chunk)
    for _ in range(2):
        _nometa()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    c0.record(stream)
    for _ in range(reps):
        _nometa()
    c1.record(stream)
    torch.cuda.synchronize()
    nometa_ms = c0.elapsed_time(c1) / reps
    kernels["without_meta_comparator"] = {
        "avg_ms": nometa_ms, "head_tokens_per_s": B * H * T / (nometa_ms / 1e3),
        "palimpsa_forward_over_comparator": fwd_avg_ms / nometa_ms,
        "note": "same scan inputs with the importance frozen at I_prior (Mamba2 / scalar-decay form), "
                "same time-split plan as the forward; timed after the timed region"}

    # The fused prologue (palimpsa_forward_fused / palimpsa_step_fused): the same
    # workload from raw projections with the Palimpsa-D q/k norm and the v* input,
    # timed outside the timed region against the unfused kernels above.
    raw = syn.sequence_inputs(wl, device=dev, seed=seed, raw=True)

    def _fused():
        pal.palimpsa_forward_fused(raw["q"], raw["k"], raw["v"], raw["beta_raw"], raw["d_raw"], raw["A"],
                                   raw["I_prior"], raw["b_scale"], qk_norm=True, v_star=True, y=y_pre, mu_T=mu,
                                   I_T=I, chunk=wl.chunk)
    for _ in range(2):
        _fused()
    c0.record(stream)
    for _ in range(reps):
        _fused()
    c1.record(stream)
    torch.cuda.synchronize()
    fused_ms = c0.elapsed_time(c1) / reps
    kernels["palimpsa_fwd_fused"] = {
        "avg_ms": fused_ms, "head_tokens_per_s": B * H * T / (fused_ms / 1e3), "over_unfused": fused_ms / fwd_avg_ms,
        "note": "raw q, k, v*, beta_raw, d_raw in; softplus, b_scale * sigmoid and the q/k L2 norm applied while "
                "staging; timed after the timed region"}
    if S:
        SF = min(S, 64)
        rdec = syn.decode_inputs(wl, SF, device=dev, seed=seed, raw=True)

        def _fused_steps():
            # the SF tokens in order, enqueued by one palimpsa_step_sequence_fused call
            pal.palimpsa_step_fused(rdec["q"], rdec["k"], rdec["v"], rdec["beta_raw"], rdec["d_raw"], raw["A"],
                                    raw["I_prior"], mu, I, raw["b_scale"], qk_norm=True, v_star=True, y=y_dec[:SF])
        _fused_steps()
        c0.record(stream)
        _fused_steps()
        c1.record(stream)
        torch.cuda.synchronize()
        fstep_ms = c0.elapsed_time(c1) / SF
        db = decode_step_bytes(B, H, dk, dv, in_bytes)
        kernels["palimpsa_step_fused"] = {
            "avg_ms": fstep_ms, "hbm_gbs": db / (fstep_ms / 1e3) / 1e9,
            "frac_of_hbm_peak": db / (fstep_ms / 1e3) / 1e9 / hbm_peak,
            "over_unfused": fstep_ms / kernels["palimpsa_step"]["avg_ms"],
            "note": f"{SF} fused steps from raw inputs; timed after the timed region"}

    # Variable-length batch: the same tokens per head packed as 4 B ragged
    # sequences (seeded uniform length mix), timed against the dense forward.
    if not S:
        lengths = syn.varlen_lengths(B * T, 4 * B, seed)
        pk = syn.packed_inputs(wl, lengths, H=H, device=dev, seed=seed)
        mx = max(lengths)
        yv = torch.empty((H, B * T, dv), dtype=f32, device=dev)
        mv = torch.empty((len(lengths), H, dv, dk), dtype=f32, device=dev)
        Iv = torch.empty_like(mv)

        def _varlen():
            pal.palimpsa_forward_varlen(pk["q"], pk["k"], pk["v"], pk["beta"], pk["d_t"], pk["A"], pk["I_prior"],
                                        pk["cu_seqlens"], max_seqlen=mx, y=yv, mu_T=mv, I_T=Iv, chunk=wl.chunk)
        for _ in range(2):
            _varlen()
        c0.record(stream)
        for _ in range(reps):
            _varlen()
        c1.record(stream)
        torch.cuda.synchronize()
        var_ms = c0.elapsed_time(c1) / reps
        kernels["palimpsa_fwd_varlen"] = {
            "avg_ms": var_ms, "head_tokens_per_s": B * H * T / (var_ms / 1e3), "over_dense": var_ms / fwd_avg_ms,
            "sequences": len(lengths), "max_seqlen": mx,
            "note": "the dense workload's tokens per head packed as ragged sequences; timed after the timed region"}

    # The backward through the scan (gradients of <dy, y> for every input), timed
    # outside the timed region on the same inputs.
    if not S:
        dy = torch.randn((B, H, T, dv), dtype=f32, device=dev)
        def _bwd():
            pal.palimpsa_backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"], inp["I_prior"],
                                  None, None, dy, want_state_grads=False)
        _bwd()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(3):
            _bwd()
        b1.record(stream)
        torch.cuda.synchronize()
        bwd_ms = b0.elapsed_time(b1) / 3
        # the training pair: a forward that writes the 32-token checkpoints, and the
        # backward that reads them instead of recomputing them
        ck = pal.palimpsa_forward_checkpointed(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"],
                                               inp["I_prior"], y=y_pre, mu_T=mu, I_T=I, chunk=wl.chunk)[3]
        b0.record(stream)
        for _ in range(3):
            pal.palimpsa_forward_checkpointed(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"],
                                              inp["I_prior"], y=y_pre, mu_T=mu, I_T=I, ckpt=ck, chunk=wl.chunk)
        b1.record(stream)
        torch.cuda.synchronize()
        fwd_ck_ms = b0.elapsed_time(b1) / 3

        def _bwd_ck():
            pal.palimpsa_backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d_t"], inp["A"], inp["I_prior"],
                                  None, None, dy, want_state_grads=False, ckpt=ck)
        _bwd_ck()
        b0.record(stream)
        for _ in range(3):
            _bwd_ck()
        b1.record(stream)
        torch.cuda.synchronize()
        bwd_ck_ms = b0.elapsed_time(b1) / 3
        del ck
        # the same training pair over the packed ragged batch of the varlen line
        dyv = torch.randn((H, B * T, dv), dtype=f32, device=dev)
        ckv = pal.palimpsa_forward_varlen_checkpointed(pk["q"], pk["k"], pk["v"], pk["beta"], pk["d_t"], pk["A"],
                                                       pk["I_prior"], pk["cu_seqlens"], max_seqlen=mx, y=yv,
                                                       mu_T=mv, I_T=Iv, chunk=wl.chunk)[3]

        def _pair_varlen():
            pal.palimpsa_forward_varlen_checkpointed(pk["q"], pk["k"], pk["v"], pk["beta"], pk["d_t"], pk["A"],
                                                     pk["I_prior"], pk["cu_seqlens"], max_seqlen=mx, ckpt=ckv, y=yv,
                                                     mu_T=mv, I_T=Iv, chunk=wl.chunk)
            pal.palimpsa_backward_varlen(pk["q"], pk["k"], pk["v"], pk["beta"], pk["d_t"], pk["A"], pk["I_prior"],
                                         pk["cu_seqlens"], None, None, dyv, max_seqlen=mx, want_state_grads=False,
                                         ckpt=ckv)
        _pair_varlen()
        b0.record(stream)
        for _ in range(3):
            _pair_varlen()
        b1.record(stream)
        torch.cuda.synchronize()
        pair_var_ms = b0.elapsed_time(b1) / 3
        del ckv, dyv
        kernels["palimpsa_train_pair_varlen"] = {
            "avg_ms": pair_var_ms, "head_tokens_per_s": B * H * T / (pair_var_ms / 1e3),
            "over_dense_pair": pair_var_ms / (fwd_ck_ms + bwd_ck_ms), "sequences": len(lengths), "max_seqlen": mx,
            "note": "checkpointed packed forward + packed backward from its checkpoints over the varlen line's "
                    "ragged batch; timed after the timed region"}
        fp32_peak = n_sms * rates["ffma"] * sm_max * 1e6 / BWD_MIN_FP32_OPS / 1e9  # G element-tokens/s
        bwd_rate = {name: E_fwd / (ms / 1e3) / 1e9 for name, ms in (("recomputing", bwd_ms),
                                                                      ("from_checkpoints", bwd_ck_ms))}
        kernels["palimpsa_backward"] = {
            "avg_ms": bwd_ms, "head_tokens_per_s": B * H * T / (bwd_ms / 1e3),
            "over_forward": bwd_ms / fwd_avg_ms,
            "checkpointed_forward_ms": fwd_ck_ms,
            "from_checkpoints_ms": bwd_ck_ms,
            "sfu": {"achieved": bwd_rate, "peak": alu_peak, "unit": "G element-tokens/s",
                    "frac": {k: v / alu_peak for k, v in bwd_rate.items()}},
            "fp32": {"achieved": bwd_rate, "peak": fp32_peak, "unit": "G element-tokens/s",
                     "frac": {k: v / fp32_peak for k, v in bwd_rate.items()},
                     "ops_per_element_token": BWD_MIN_FP32_OPS,
                     "peak_source": f"{n_sms} SMs x {rates['ffma']:.1f} FP32 FMA/clk/SM (probe) x {sm_max:.0f} MHz "
                                    f"/ {BWD_MIN_FP32_OPS} ops"},
            "note": "gradients of <dy, y> w.r.t. q, k, v, beta, d_t, A, I_prior; "
                    "from_checkpoints: reading the states a checkpointed forward "
                    "wrote; timed after the timed region"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, inp, dec, dev, pal, ws)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": _describe(wl), "B": B, "H": H, "T_prefill": T, "decode_steps": S, "d_k": dk,
                       "d_v": dv, "inputs": "bf16" if wl.bf16 else "f32", "state": "f32",
                       "head_tokens_per_step": head_tokens,
                       "l2": "inputs larger than L2 (state alone is %.0f MB)" % (B * H * dv * dk * 8 / 1e6),
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (fwd_launches + S) * args.steps, "clocks": clocks,
            "issue_rates_per_clk_per_sm": rates,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def issue_rates(pal):
    """Instructions per clock and SM of the SFU reciprocal, the SFU 2^x and the FP32 FMA,
    measured on this GPU by the library's probe (one CTA per SM, SM cycle counter)."""
    return {op: pal.palimpsa_probe_issue_rate(op) for op in ("rcp", "ex2", "ffma")}


def run_probe_rates(local):
    import torch

    import metaplastic_linear_attention_gb300 as pal
    from metaplastic_linear_attention_gb300 import build_lib
    torch.cuda.set_device(local)
    build_lib.build()
    pal.load_library()
    props = torch.cuda.get_device_properties(local)
    peaks, kind = _measured_peaks()
    reps = [{op: pal.palimpsa_probe_issue_rate(op) for op in pal.binding.PROBE_OPS} for _ in range(5)]
    med = {op: statistics.median(r[op] for r in reps) for op in reps[0]}
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    print(json.dumps({"gpu": props.name, "sms": props.multi_processor_count, "per_clk_per_sm_runs": reps,
                      "per_clk_per_sm_median": med, "sm_max_mhz": sm_max,
                      "rcp_peak_G_per_s": props.multi_processor_count * med["rcp"] * sm_max / 1e3}), flush=True)


def _workload(args):
    from metaplastic_linear_attention_gb300 import synthetic as syn
    wl = syn.WORKLOADS[args.workload]
    over = {k: v for k, v in (("B", args.B), ("H", args.H), ("T", args.T), ("steps", args.decode_steps))
            if v is not None}
    return wl.with_(**over) if over else wl


def _describe(wl):
    if wl.steps:
        return (f"{wl.name}: B={wl.B} H={wl.H} d_k={wl.d_k} d_v={wl.d_v}, {wl.T}-token chunked prefill + "
                f"{wl.steps} decode steps, {'bf16' if wl.bf16 else 'fp32'} inputs, fp32 state")
    return (f"{wl.name}: B={wl.B} H={wl.H} T={wl.T} d_k={wl.d_k} d_v={wl.d_v}, chunked forward, "
            f"{'bf16' if wl.bf16 else 'fp32'} inputs, fp32 state")


def run_e2e(args, wl, inp, dec, dev, pal, ws):
    """Same job through the public calls with pinned HOST inputs and outputs:
    every step copies its inputs host->device and its y device->host."""
    import torch
    import torch.distributed as dist

    B, H, T, dk, dv, S = wl.B, wl.H, wl.T, wl.d_k, wl.d_v, wl.steps
    h_inp = {k: v.to("cpu").pin_memory() for k, v in inp.items()}
    h_dec = {k: v.to("cpu").pin_memory() for k, v in dec.items()} if S else None
    h_ypre = torch.empty((B, H, T, dv), dtype=torch.float32, pin_memory=True)
    h_ydec = torch.empty((max(S, 1), B, H, dv), dtype=torch.float32, pin_memory=True)
    mu = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    I = torch.empty_like(mu)

    def one_step():
        pal.palimpsa_forward_chunked(h_inp["q"], h_inp["k"], h_inp["v"], h_inp["beta"], h_inp["d_t"], h_inp["A"],
                                     h_inp["I_prior"], y=h_ypre, mu_T=mu, I_T=I, chunk=wl.chunk)
        if S:
            pal.palimpsa_step(h_dec["q"], h_dec["k"], h_dec["v"], h_dec["beta"], h_dec["d_t"], h_inp["A"],
                              h_inp["I_prior"], mu, I, y=h_ydec[:S])

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t0, ws, dev)
    h2d = sum(v.numel() * v.element_size() for v in h_inp.values())
    h2d += 2 * H * 4 if S else 0  # A and I_prior go again with the decode call
    if S:
        h2d += sum(v.numel() * v.element_size() for v in h_dec.values())
    d2h = h_ypre.numel() * 4 + (S * B * H * dv * 4 if S else 0)
    value = whole_job_rate(B * H * (T + S), ws, el / args.steps)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": el / args.steps * 1e3, "timer": "host wall clock around device-synchronised steps",
            "pipeline": "host buffers streamed in blocks: copies in, kernels, copies out on three streams"}


# ----------------------------------------------------------------------------- the oracle (CPU baseline)

def _oracle_sample(wl, n_heads, seed=12345):
    """A bounded sample of the workload for the fp64 oracle: n_heads heads over the
    whole token stream (prefill followed by the decode tokens, which the oracle
    treats as one continuous scan: a decode step is one token of the recurrence)."""
    import numpy as np
    import torch

    from metaplastic_linear_attention_gb300 import synthetic as syn
    Ttot = wl.T + wl.steps
    sub = wl.with_(B=1, H=n_heads, T=Ttot, steps=0)
    x = syn.sequence_inputs(sub, seed=seed)
    f = syn.as_float64_numpy
    return [f(x[k]) for k in ("q", "k", "v", "beta", "d_t", "A", "I_prior")], n_heads * Ttot


def cpu_baseline(wl, seconds):
    import oracle
    threads = oracle.max_threads()
    args1, ht1 = _oracle_sample(wl, 1)
    t0 = time.perf_counter()
    oracle.forward(*args1)
    t1 = time.perf_counter() - t0
    n = max(1, min(wl.B * wl.H, int(seconds / max(t1, 1e-3))))
    args_n, ht = _oracle_sample(wl, n)
    t0 = time.perf_counter()
    oracle.forward(*args_n)
    el = time.perf_counter() - t0
    return {"value": ht / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} head(s) x {wl.T + wl.steps} tokens (d_k={wl.d_k}, d_v={wl.d_v}) of the {wl.name} "
                      f"workload, fp64 C oracle, {el:.1f} s"}


def run_reference(args, ws, rank):
    """--impl reference: the fp64 CPU oracle on the host cores, on a bounded sample of
    the same workload per step (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    wl = _workload(args)
    oracle.build()
    threads = oracle.max_threads()
    args1, _ = _oracle_sample(wl, 1)
    t0 = time.perf_counter()
    oracle.forward(*args1)
    t1 = time.perf_counter() - t0
    per_step = max(0.5, min(args.ref_step_seconds, 150.0 / max(1, args.steps + args.warmup)))
    n = max(1, min(wl.B * wl.H, int(per_step / max(t1, 1e-3))))
    sample, ht = _oracle_sample(wl, n)
    for _ in range(args.warmup):
        oracle.forward(*sample)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(*sample)
        times.append(time.perf_counter() - t0)
    el = sum(times)
    value = ht * args.steps / el
    desc = (f"{n} head(s) x {wl.T + wl.steps} tokens of the {wl.name} workload per step, fp64 C oracle "
            f"({threads} threads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _describe(wl), "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="decode",
                   choices=["decode", "small_layer", "layer_760m", "long_context", "tiny"])
    p.add_argument("--B", type=int, default=None, help="override the workload's batch (profiling cases)")
    p.add_argument("--H", type=int, default=None, help="override the workload's heads")
    p.add_argument("--T", type=int, default=None, help="override the workload's scan length")
    p.add_argument("--decode-steps", type=int, default=None, help="override the decode step count")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time for cpu_baseline")
    p.add_argument("--ref-step-seconds", type=float, default=4.0)
    p.add_argument("--probe-rates", action="store_true",
                   help="only measure the SFU / FMA issue rates per clock and SM, print them and exit")
    p.add_argument("--traffic", type=float, default=None,
                   help="DRAM bytes per launch of the dominant kernel from an ncu capture (else null)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.gpus < 1:
        p.error("--gpus must be >= 1")
    launched = "WORLD_SIZE" in os.environ
    if launched and int(os.environ["WORLD_SIZE"]) != args.gpus:
        p.error(f"--gpus {args.gpus} disagrees with WORLD_SIZE={os.environ['WORLD_SIZE']} set by the launcher")
    if args.probe_rates:
        run_probe_rates(_dist_env()[2])
        return
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone does the work (in this process when no launcher started ranks)
        ws, rank, _ = _dist_env()
        run_reference(args, args.gpus, rank)
        return
    if not launched and args.gpus > 1:
        # no launcher: start one rank per GPU here, each an independent replica
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            raise SystemExit(f"bench: --gpus {args.gpus} needs {args.gpus} visible GPUs, found {have}")
        spawn_ranks(args.gpus, _run_rank, (list(argv) if argv is not None else sys.argv[1:],))
        return
    ws, rank, local = _dist_env()
    run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
