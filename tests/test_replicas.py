"""The multi-GPU path of bench.py (replicas, no data exchange) on CPU ranks.

The step shards by sequence with no exchange, so N GPUs run N independent
replicas: each rank draws its own inputs and the job's throughput is the
total steps over the slowest rank's time. Two gloo ranks on the host check
that aggregation and the per-rank seeding.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from medusa_speculative_decoding_heads_gb300 import configs, synth

        local_ms = 10.0 + 5.0 * rank   # rank 1 is the slow one
        ms, value = bench.replica_throughput(local_ms, steps=4, world=world, device="cpu")
        w = configs.scaled(configs.get("tiny_fp32"), L_range=(16, 32))
        si = synth.make_step_inputs(w, seed=bench.replica_seed(7, rank), device="cpu")
        h = si.h.double()
        hs = [torch.zeros_like(h) for _ in range(world)]
        dist.all_gather(hs, h)
        out[rank] = (ms, value, bool(torch.equal(hs[0], hs[1])))
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        ms, value, same_inputs = out[rank]
        assert ms == pytest.approx(15.0)                      # the slowest rank's time, on every rank
        assert value == pytest.approx(world * 4 / 0.015)      # total steps of all ranks over that time
        assert not same_inputs                                # replicas do not repeat each other's work


def test_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.replica_throughput(20.0, steps=10, world=1, device="cpu")
    assert ms == 20.0 and value == pytest.approx(500.0)
    assert bench.replica_seed(3, 0) == 3 and bench.replica_seed(3, 1) != 3


def test_gpus_flag_must_match_the_launcher():
    """`--gpus 2` under a launcher that started a different number of ranks is refused
    before any GPU work."""
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "--gpus 2" in r.stderr


def test_gpus_flag_starts_the_replicas(monkeypatch):
    """`--gpus 4` run plainly re-launches the script as 4 ranks under torch.distributed.run."""
    sys.path.insert(0, ROOT)
    import bench

    seen = {}
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "3"])
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: seen.setdefault("cmd", cmd) and 0)
    assert bench.main() == 0
    cmd = seen["cmd"]
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "3"]
