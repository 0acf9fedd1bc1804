"""The multi-GPU path of bench.py is replicas only (no collective on the data
path); its host logic -- slowest-rank timing, whole-job value, rank 0 alone
printing the reference line -- is checked here with two gloo ranks on CPU."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 2.0 + 3.0 * rank
        ms_max = bench.max_over_ranks(local_ms, dist)
        bench.barrier(dist)
        args = type("A", (), dict(workload="mha_b1_h2_s128_d64_fp16", warmup=1, steps=1,
                                  gpus=world))()
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args)
        out[rank] = (ms_max, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_timing_and_reference_line():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0][0] == out[1][0] == 5.0  # both ranks see the slowest rank's time
    line = json.loads(out[0][1])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert out[1][1] == ""  # only rank 0 prints


def test_replica_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.replica_value(2.0e12, 2.0, 1)
    assert abs(one - 1000.0) < 1e-9
    assert abs(bench.replica_value(2.0e12, 2.0, 4) - 4 * one) < 1e-9
