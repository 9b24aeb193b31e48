"""bench.py's multi-rank host logic on CPU: two gloo ranks, replicas of the step.

The step does not shard (each GPU runs its own replica), so the only cross-rank work
is the barrier around the timed region and the max over ranks of the elapsed time.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, steps, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms, value = bench.combine_ranks(ms_by_rank[rank], steps, world, torch.device("cpu"))
        dist.barrier()
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ms_by_rank", [(10.0, 25.0), (40.0, 12.5)])
def test_two_ranks_take_the_slowest(ms_by_rank):
    world, steps = 2, 400
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), ms_by_rank, steps, out), nprocs=world,
                       start_method="spawn", join=True)
    slow = max(ms_by_rank)
    for r in range(world):
        ms, value = out[r]
        assert ms == slow
        # whole-job throughput: both replicas' steps over the slowest rank's time
        assert value == pytest.approx(world * steps / (slow / 1e3))


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.combine_ranks(8.0, 100, 1, torch.device("cpu"))
    assert ms == 8.0 and value == pytest.approx(100 / 0.008)


def test_reference_arm_other_ranks_print_nothing(monkeypatch, capsys):
    """Under torchrun only rank 0 runs the oracle arm; the others exit without work."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "0"])
    bench.run_reference(bench.parse_args())
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    """Rank 0's oracle line carries the contract's keys (1B-shaped one-row workload, one step)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                                      "--workload", "1b-1"])
    bench.run_reference(bench.parse_args())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
