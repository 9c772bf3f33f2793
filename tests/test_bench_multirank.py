"""Host logic of bench.py's multi-process (replica) path, on CPU with the gloo backend.

Under torchrun every rank runs one full replica of the step; the job's time is the
slowest rank's, and the whole-job value counts the work of all ranks. These tests run
two gloo ranks on 127.0.0.1 and check that reduction, and that the reference arm runs on
rank 0 alone.
"""
import contextlib
import io
import json
import os
import socket
import sys
import types

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank times differ; every rank must see the element-wise maximum
        mx = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 3.0])
        dist.barrier()
        rate = bench.whole_job_rate(2.0e12, mx[0], world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": mx, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        res = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert res["max"] == [11.0, 5.0, 3.0]
        # two ranks did 2e12 units each; the job took 11 ms (the slower rank)
        assert res["rate"] == pytest.approx(2 * 2.0e12 / 11e-3)


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_rate(1.0e9, 2.0, 1) == pytest.approx(5.0e11)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = types.SimpleNamespace(steps=3, warmup=3, ref_seconds=1.0)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args)  # rank 1: returns at once, prints nothing
    assert buf.getvalue() == ""
