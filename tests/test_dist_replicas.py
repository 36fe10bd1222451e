"""The N > 1 path on CPU: two gloo ranks, each with its own batch, timing
reduced by max over ranks, whole-job throughput over all ranks.  No GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, make_batch
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = WORKLOADS["bypass_b16_l256"]
    hb = make_batch(wl, seed=bench.rank_seed(wl.seed, rank))
    # each rank's batch is its own; the step time is the slowest rank's
    fake_ms = 1.0 + rank
    ms = bench.reduce_max(fake_ms, dist, torch.device("cpu"))
    digest = float(hb["q"].float().sum())
    all_d = [None] * world
    dist.all_gather_object(all_d, digest)
    out[rank] = (ms, bench.job_throughput(hb["B"] * hb["S"], world, ms), all_d)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_weak_scaling_on_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (ms0, v0, d0), (ms1, v1, d1) = out[0], out[1]
    assert ms0 == ms1 == 2.0                     # max over ranks
    assert v0 == v1 == 16 * 2 / 2.0e-3           # all ranks' queries / slowest time
    assert d0 == d1 and d0[0] != d0[1]           # the two ranks decode different batches


def test_single_rank_reduction_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, None, None) == 3.5
    assert bench.rank_seed(1003, 0) == 1003 and bench.rank_seed(1003, 1) != 1003
