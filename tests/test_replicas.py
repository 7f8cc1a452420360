"""The multi-GPU path of bench.py is replicas only: every rank streams its own
copy of the base, no collective touches the data path, and the job's rate is
the units of all ranks over the slowest rank's time.  These tests run that
logic as two gloo ranks on the CPU."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, local_seconds):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        t_max = bench.max_over_ranks_of(local_seconds[rank], world, "cpu")
        rate = bench.whole_job_rate(1024 * 10, world, t_max)
        bench.rank_barrier(world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t_max": t_max, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    import tempfile
    world, secs = 2, [1.25, 2.5]
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_rank_main, args=(world, _free_port(), d, secs), nprocs=world, join=True)
        res = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(world)]
    for r in res:
        assert r["t_max"] == max(secs)                       # every rank sees the slowest time
        assert r["rate"] == world * 1024 * 10 / max(secs)    # whole-job units over that time


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks_of(3.0, 1, "cpu") == 3.0
    bench.rank_barrier(1)
    assert bench.whole_job_rate(1024, 1, 0.5) == 2048


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the oracle arm prints one line from rank 0; other ranks exit without work."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = type("A", (), dict(workload="attn8b", gpus=2, steps=1, warmup=3))()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_every_workload_names_its_config(name):
    w = bench.WORKLOADS[name]
    assert w["name"] and w["kind"] in ("stack", "layer", "attn", "ce") and w["M"] > 0
