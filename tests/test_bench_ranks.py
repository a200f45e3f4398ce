"""The multi-process side of bench.py on CPU: two gloo ranks, each an
independent replica, reduce their step times to the slowest rank's and report
the units of all ranks over that time (weak scaling, no data-path collective)."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r was slower on the step, faster on the end-to-end leg
    step_s, e2e_s = bench.reduce_over_ranks(torch, [0.5 + rank, 3.0 - rank], "cpu")
    tput = bench.job_throughput(8192, world, step_s)
    with open(os.path.join(result_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{step_s} {e2e_s} {tput}")
    dist.barrier()
    dist.destroy_process_group()


def test_single_process_is_identity():
    import bench
    assert bench.reduce_over_ranks(torch, [1.25, 2], "cpu") == [1.25, 2.0]
    assert bench.job_throughput(8192, 1, 0.5) == 16384


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    got = [tuple(map(float, open(tmp_path / f"r{r}.txt").read().split())) for r in range(world)]
    for step_s, e2e_s, tput in got:
        assert step_s == 1.5            # max over ranks of 0.5 + rank
        assert e2e_s == 3.0             # max over ranks of 3 - rank
        assert tput == 8192 * 2 / 1.5   # both replicas' tokens over the slowest time


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the reference arm (the oracle on host cores) runs and
    prints on rank 0 only; every other rank exits 0 without work or output."""
    import argparse
    import bench
    args = argparse.Namespace(workload="tiny_f32", steps=1, warmup=0)
    assert bench.reference_arm(args, 2, 1) == 0
    assert capsys.readouterr().out == ""
    assert bench.reference_arm(args, 2, 0) == 0
    line = capsys.readouterr().out.strip().splitlines()[-1]
    import json
    d = json.loads(line)
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
