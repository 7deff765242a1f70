"""Host logic of the multi-GPU benchmark path, run as world_size-2 gloo ranks on CPU.

The path shards by independent heads: every rank runs its own replica (no data-path
collective); only the timing is combined, as the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        worst = bench.max_over_ranks(local_ms, ws)
        dist.barrier()
        seed = bench.replica_seed(20264, rank)
        from metaplastic_linear_attention_gb300 import synthetic as syn
        x = syn.sequence_inputs(syn.WORKLOADS["tiny"].with_(T=8), seed=seed)["q"]
        out[rank] = (worst, seed, float(x.sum()), bench.whole_job_rate(1000, ws, worst / 1e3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_as_the_slowest_and_run_independent_replicas():
    ws = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn", join=True)
    (w0, s0, x0, r0), (w1, s1, x1, r1) = out[0], out[1]
    assert w0 == w1 == 15.0                 # both ranks report the max over ranks
    assert s0 != s1 and x0 != x1            # independent replicas: different seeded inputs
    assert r0 == r1 == pytest.approx(1000 * 2 / 0.015)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(12_582_912, 1, 0.18) == pytest.approx(12_582_912 / 0.18)
    assert bench.replica_seed(5, 0) == 5
