"""Two-rank (gloo, CPU) checks of the multi-GPU plumbing of bench.py.

On N GPUs the decode runs as N independent replicas (one process per GPU, no
collective on the data path): the only cross-rank steps are the barriers
around the timed region and the max over ranks of the measured time, from
which the whole-job throughput is computed. These run here as two gloo ranks.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    bench.init_dist(w)
    assert torch.distributed.get_backend() == "gloo"
    bench.barrier(w)
    # each rank timed its own replica; the job is as slow as the slowest rank
    my_seconds = [1.5, 2.5][rank]
    slowest = bench.max_over_ranks(my_seconds, w, torch.device("cpu"))
    value = bench.job_value(w, 65536, 10, slowest)
    ref = bench.run_reference(type("A", (), {"workload": "tiny_fp32", "warmup": 0, "steps": 1,
                                             "cpu_seconds": 0.2})(), r, w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "slowest": slowest, "value": value,
                   "ref_none": ref is None, "ref_value": None if ref is None else ref["value"]}, f)
    bench.barrier(w)
    torch.distributed.destroy_process_group()


def test_two_ranks_barrier_max_and_job_value(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["slowest"] == 2.5                      # max over ranks, seen by every rank
        assert d["value"] == pytest.approx(world * 65536 * 10 / 2.5)
    # the oracle arm runs on rank 0 only; the other ranks exit without work
    assert res[0]["ref_none"] is False and res[0]["ref_value"] > 0
    assert res[1]["ref_none"] is True


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.job_value(1, 100, 4, 2.0) == pytest.approx(200.0)
