"""Host logic of the multi-GPU bench path, on CPU ranks (gloo, world size 2):
every rank draws its own batch of the same shape (weak scaling, no exchange
between ranks) and the step time reported is the slowest rank's."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench
from quantized_kv_cache_kvarn_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.0 + 0.5 * rank
        worst = bench.max_over_ranks(ms, "cpu")
        wl = W.WORKLOADS["toy"].with_(num_seqs=2, context=300)
        case = W.make_dense(wl, device="cpu", seed=bench.rank_seed(wl.seed, rank))
        sums = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([case.q.double().sum(), case.k.double().sum()]))
        out[rank] = (worst, [tuple(x.tolist()) for x in sums], tuple(case.q.shape))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks():
    world = 2
    with tmp.Manager() as mgr:
        out = mgr.dict()
        tmp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        worst, sums, shape = res[r]
        assert worst == 1.5  # the slower rank's time, on every rank
        assert sums[0] != sums[1]  # different batches
        assert shape == res[0][2]  # of the same shape
    assert res[0][1] == res[1][1]


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.rank_seed(1000, 0) == 1000 and bench.rank_seed(1000, 1) != 1000
