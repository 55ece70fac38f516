"""The multi-rank (replica) logic of bench.py on CPU with gloo, world size 2:
whole-job throughput = bytes of all ranks / slowest rank's time, and every
rank draws an independent instance of the workload."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    # rank 0: 100 MB in 2 ms, rank 1: 300 MB in 5 ms -> 400 MB / 5 ms
    b, ms = (100e6, 2.0) if rank == 0 else (300e6, 5.0)
    ms_max, gbs = bench.job_throughput(dist, b, ms, "cpu")
    w = bench.make_workload("gqa_bf16", "cpu", rank)
    w_ref = bench.make_workload("gqa_bf16", "cpu", 0)
    out[rank] = (ms_max, gbs, bool(torch.equal(w.q, w_ref.q)))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_two_ranks_gloo():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in (0, 1):
        ms_max, gbs, same = out[rank]
        assert ms_max == 5.0
        assert gbs == pytest.approx(400e6 / 5e-3 / 1e9)
        assert same == (rank == 0)     # replicas draw independent workloads


def test_job_throughput_single_process():
    import bench
    ms, gbs = bench.job_throughput(None, 553e6, 0.1, "cpu")
    assert ms == 0.1 and gbs == pytest.approx(5530.0)
