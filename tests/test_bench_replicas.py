"""bench.py's replica harness on CPU: two gloo ranks, the max-over-ranks timing and the
whole-job throughput it feeds (the GPU ranks use the same functions over NCCL)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    ws, r, local = bench._dist()
    assert (ws, r, local) == (2, rank, rank)
    bench._barrier(ws)
    ms = [12.5, 40.0][rank]                       # the slower replica sets the job time
    out[rank] = bench._max_over_ranks(ws, ms, "cpu")
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(port, out), nprocs=2, join=True)
        assert dict(out) == {0: 40.0, 1: 40.0}


def test_whole_job_throughput_counts_every_replica():
    import bench
    # 2 replicas x 8 requests x 15 drafts x 20 steps in 40 ms
    assert bench._throughput(2, 8, 15, 20, 40.0) == pytest.approx(2 * 8 * 15 * 20 / 0.040)
    assert bench._throughput(1, 8, 15, 20, 40.0) * 2 == bench._throughput(2, 8, 15, 20, 40.0)
