"""The bench's multi-process path on CPU: two gloo ranks (world size 2).

The operator shards over independent (batch, head) pairs with no exchange
step, so under torchrun each rank runs the same per-GPU workload (replicas)
and the only cross-rank operations are the timing barrier and the
max-over-ranks reduction of the measured time.  These run here as gloo ranks
on the host; the job's throughput is every rank's units over the slowest
rank's time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        seconds = 1.0 + 0.25 * r            # rank 1 is the slow one
        slowest = bench.max_over_ranks(seconds, w)
        bench.barrier(w)
        out[r] = (r, w, local, slowest, bench.job_throughput(w, 1000.0, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as manager:
        out = manager.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r, (rank, w, local, slowest, value) in res.items():
        assert (rank, w, local) == (r, world, r)
        assert slowest == pytest.approx(1.25)
        assert value == pytest.approx(2 * 1000.0 / 1.25)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(1, 10.0, 2.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun only rank 0 times the oracle and prints its line; any
    other rank returns at once without work."""
    import argparse
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None
    assert capsys.readouterr().out == ""


def test_gpus_flag_launches_replica_ranks():
    """``--gpus 2`` outside torchrun makes the bench re-run itself as two
    ranks under torchrun (rendezvous on 127.0.0.1), each with its own rank
    environment; the ranks here run the CPU stand-in of the GPU legs on gloo,
    and rank 0 alone prints one line with n_gpus = 2 and the slowest rank's
    time."""
    import json
    import subprocess
    import sys
    from pathlib import Path
    stub = Path(__file__).with_name("bench_rank_stub.py")
    res = subprocess.run([sys.executable, str(stub), "--gpus", "2", "--steps", "3",
                          "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["local_rank"] == 0
    assert line["seconds"] >= 0.1  # the slow rank's sleep
    assert line["value"] == pytest.approx(2 * 3000.0 / line["seconds"])
