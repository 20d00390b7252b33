"""Multi-process (gloo, world size 2, CPU) checks of the benchmark's N > 1 host logic.

Each GPU runs an independent replica of the reduce (no cross-GPU step), so
the only multi-rank logic is the timing aggregation: the slowest rank's time
and the sum of all ranks' bytes.  These run as two CPU processes.
"""

import os
import socket

import pytest
import torch.multiprocessing as tmp

from conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        elapsed = 1.0 + rank          # rank 1 is the slower one
        units = 100.0 * (rank + 1)
        t, u = bench.aggregate_over_ranks(elapsed, units)
        bench.barrier()
        results[rank] = (t, u)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = tmp.get_context("spawn").Manager()
    results = mgr.dict()
    tmp.start_processes(_worker, args=(world, port, results), nprocs=world, join=True,
                        start_method="spawn")
    assert results[0] == results[1] == (2.0, 300.0)


def test_aggregate_is_identity_without_a_group():
    import bench
    assert bench.aggregate_over_ranks(1.5, 42.0) == (1.5, 42.0)


def test_rotation_sets_exceed_l2():
    import bench
    l2 = 126 * 2**20
    for set_bytes in (786_432, 2_359_296, 67_108_864, 2_415_919_104):
        R = bench.rotation_sets(set_bytes, l2)
        assert R * set_bytes > bench.ROTATE_FACTOR * l2 or R == 4096
    assert bench.rotation_sets(10 * l2, l2) == 1   # one set already exceeds 3x L2


@pytest.mark.parametrize("steps", [1, 7])
def test_reference_arm_prints_one_line(steps, capsys):
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", str(steps), "--warmup", "3"])
    line = capsys.readouterr().out.strip().splitlines()
    assert len(line) == 1
    rec = json.loads(line[0])
    assert rec["impl"] == "reference" and rec["steps"] == steps and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def _reference_worker(rank, world, results):
    import contextlib
    import io
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    results[rank] = buf.getvalue()


def test_reference_arm_prints_on_rank_0_only():
    world = 2
    mgr = tmp.get_context("spawn").Manager()
    results = mgr.dict()
    tmp.start_processes(_reference_worker, args=(world, results), nprocs=world, join=True,
                        start_method="spawn")
    import json
    lines = results[0].strip().splitlines()
    assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"
    assert json.loads(lines[0])["n_gpus"] == world
    assert results[1] == ""
