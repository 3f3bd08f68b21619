"""The benchmark's multi-rank host logic on CPU with two gloo ranks (no GPU):
under torchrun every rank times its own replica of the layer, the step time is
the maximum over ranks, the whole-job throughput counts every rank's layer,
and the reference arm runs (and prints) on rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method="tcp://127.0.0.1:%d" % port)
    import bench
    res = {"dist_init": list(bench.dist_init()),
           # rank r's step took 1 + r ms and its end-to-end step 10 - r ms
           "max": bench.max_over_ranks([1.0 + rank, 10.0 - rank])}
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_reduce_step_times_to_the_slowest(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        res = json.load(open(tmp_path / ("rank%d.json" % rank)))
        assert res["dist_init"] == [world, rank, rank]
        assert res["max"] == [2.0, 10.0]


def test_single_rank_values_pass_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 7.0]) == [3.5, 7.0]


def test_aggregate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    flops = 6.0 * 2048 * 8 * 4096 * 1536
    one = bench.aggregate_tflops(1, flops, 0.6)
    assert abs(one - flops / 0.6e-3 / 1e12) < 1e-9
    assert abs(bench.aggregate_tflops(4, flops, 0.6) - 4 * one) < 1e-9


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    args = argparse.Namespace(workload=1, steps=1, warmup=0, gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args, world=2, rank=1) == 0
    assert buf.getvalue() == ""
