"""Replica bookkeeping of bench.py on two CPU ranks (gloo): the job time is the
slowest rank's, and the whole-job throughput counts every rank's bytes.  The
path has no data-path collective (replicas only), so this is all the multi-GPU
logic there is."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    got_ws, got_rank, got_local = bench.dist_env()
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        job_ms = bench.max_over_ranks(ms, ws, torch.device("cpu"))
        value = bench.job_throughput(ws, 1_000_000, job_ms / 2)   # 2 steps in the timed region
        out[rank] = (got_ws, got_rank, got_local, job_ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_job_throughput():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    for rank in range(ws):
        got_ws, got_rank, got_local, job_ms, value = res[rank]
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert job_ms == pytest.approx(15.0)          # the slowest rank
        # 2 ranks x 1 MB a step / 7.5 ms a step
        assert value == pytest.approx(2 * 1_000_000 / 7.5e-3 / 1e9)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_throughput(1, 2_000_000_000, 1000.0) == pytest.approx(2.0)
