"""Multi-rank host logic on CPU (gloo, world size 2): the benchmark's whole-job
throughput is all ranks' FLOPs over the slowest rank's time, and every rank's
batch has its own seed (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def rmax(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def rsum(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    local_s = 1.0 + rank  # rank 1 is the slow one
    local_f = 1e12 * (rank + 1)
    value, t = bench.aggregate(local_s, local_f, world, rmax, rsum)
    from synthetic_inputs import make_qkv
    x = make_qkv(1, 1, 8, 4, seed=1004 + 1000 * rank)["q"]
    gathered = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(gathered, x)
    out[rank] = (value, t, bool(torch.equal(gathered[0], gathered[1])))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, t, same = out[r]
        assert t == pytest.approx(2.0)              # slowest rank
        assert value == pytest.approx(3e12 / 2.0)   # all ranks' work / max time
        assert not same                             # per-rank batches differ


def test_single_rank_aggregation_and_flop_model():
    import bench
    v, t = bench.aggregate(2.0, 4e12, 1)
    assert (v, t) == (2e12, 2.0)
    # forward 4 B H N^2 D + backward 7 GEMMs 14 B H N^2 D, halved when causal
    assert bench.step_flops(2, 16, 4096, 128, True) == pytest.approx(18 * 2 * 16 * 4096 ** 2 * 128 / 2)
    kf = bench.kernel_flops(1, 1, 10, 8, False)
    assert kf["fwd"] + kf["bwd_dq"] + kf["bwd_dkdv"] == pytest.approx(bench.step_flops(1, 1, 10, 8, False))
    import attention_tiled_fwd_gb300 as fa
    assert fa.attention_flops(1, 1, 10, 8, True, "bwd") == pytest.approx(bench.step_flops(1, 1, 10, 8, True,
                                                                                         ("bwd",)))
