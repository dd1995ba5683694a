"""The multi-GPU path of the benchmark is N independent replicas (no exchange
step in the single-device layer): each rank times its own steps, the job's
time is the slowest rank's and its work the sum over ranks.  This checks that
reduction with two gloo ranks on the CPU."""
import json
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out_path):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    assert bench.dist_env() == (ws, rank, rank)
    # rank r: 10 + r ms timed, 20 - r ms end to end, (r + 1) TFLOP of work
    ms, ms_e2e, fl = bench.reduce_over_ranks(10.0 + rank, 20.0 - rank, (rank + 1) * 1e12, dist,
                                             "cpu")
    dist.barrier()
    if rank == 0:
        json.dump(dict(ms=ms, ms_e2e=ms_e2e, flops=fl,
                       value=bench.job_value(fl, 5, ms)), open(out_path, "w"))
    dist.destroy_process_group()


def test_replicas_reduce_max_time_and_sum_work(tmp_path):
    out = str(tmp_path / "r0.json")
    mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    r = json.load(open(out))
    assert r["ms"] == 11.0 and r["ms_e2e"] == 20.0 and r["flops"] == 3e12
    # 5 steps of 3 TFLOP in 11 ms
    assert abs(r["value"] - 3e12 * 5 / 11e-3 / 1e12) < 1e-9


def test_single_process_passes_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(1.5, 2.5, 7.0, None, "cpu") == (1.5, 2.5, 7.0)
