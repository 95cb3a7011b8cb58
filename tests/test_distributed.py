"""Multi-rank logic of bench.py on CPU (gloo, world size 2).

The round shards by sequence with no collective: every rank denoises its own batch, the
job's time is the slowest rank's, and the job's value counts every rank's positions.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], world)
        value = bench.job_value(512, world, ms_max)
        with open(f"{out_path}.{rank}", "w") as f:
            f.write(f"{ms_max!r} {value!r}\n")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    times = [0.25, 0.375]          # rank 1 is the slow one
    out = str(tmp_path / "res")
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        ms_max, value = map(float, open(f"{out}.{r}").read().split())
        assert ms_max == 0.375
        assert value == pytest.approx(512 * world / 0.375e-3, rel=1e-12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_value(512, 1, 0.25) == pytest.approx(2.048e6)


def test_rank_seeds_are_distinct_and_stable():
    seeds = [bench.rank_seed(1002, r) for r in range(8)]
    assert len(set(seeds)) == 8
    assert seeds[0] == 1002
    assert seeds == [bench.rank_seed(1002, r) for r in range(8)]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = bench.parse_args(["--impl", "reference", "--gpus", "2"])
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
