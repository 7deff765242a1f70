"""Host logic of the multi-GPU benchmark path, run as world_size-2 gloo ranks on CPU.

The path shards by independent heads: every rank runs its own replica (no data-path
collective); only the timing is combined, as the max over ranks. Without a launcher,
``bench.py --gpus N`` starts the N ranks itself (``bench.spawn_ranks``)."""
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


def _launched_rank(out_dir):
    """A rank started by bench.spawn_ranks: the environment torchrun would set, a gloo
    group built from it, and the benchmark's cross-rank timing."""
    ws, rank, local = bench._dist_env()
    assert os.environ["MASTER_ADDR"] == "127.0.0.1" and local == rank
    dist.init_process_group("gloo")
    try:
        assert dist.get_world_size() == ws and dist.get_rank() == rank
        worst = bench.max_over_ranks(20.0 + rank, ws)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ws} {rank} {worst}")
    finally:
        dist.destroy_process_group()


def _failing_rank(out_dir):
    """Rank 1 fails before the group forms; rank 0 would wait for it at the rendezvous."""
    ws, rank, _ = bench._dist_env()
    if rank == 1:
        raise RuntimeError("injected rank failure")
    dist.init_process_group("gloo")
    dist.destroy_process_group()


def test_spawned_ranks_get_the_launcher_environment_and_time_as_the_slowest(tmp_path):
    bench.spawn_ranks(2, _launched_rank, (str(tmp_path),))
    got = sorted(open(tmp_path / f"rank{r}.txt").read().split() for r in range(2))
    assert got == [["2", "0", "21.0"], ["2", "1", "21.0"]]


def test_a_failed_spawned_rank_stops_the_others_and_fails_the_run(tmp_path):
    with pytest.raises(SystemExit, match=r"rank\(s\) \[1\] of 2 failed"):
        bench.spawn_ranks(2, _failing_rank, (str(tmp_path),))


def test_gpus_beyond_the_visible_devices_fail_loudly(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(torch.cuda, "device_count", lambda: 1)
    with pytest.raises(SystemExit, match="needs 4 visible GPUs, found 1"):
        bench.main(["--gpus", "4"])


def test_gpus_must_agree_with_the_launcher(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "4"])
