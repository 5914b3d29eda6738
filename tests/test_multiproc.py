"""The multi-rank path on CPU (gloo, world size 2).

The op has no exchange step: every (batch, head) is an independent problem, so ranks
either run replicas of the workload (the benchmark's weak scaling) or own disjoint
head ranges (tensor-parallel style, each rank holding the qkv of its own heads).
These tests check the host side of both without a GPU:
  * head shards computed on separate ranks and gathered equal the single-process
    result bit for bit (no cross-head term exists to lose);
  * the benchmark's timing is the max over ranks and its throughput counts every
    rank's work over that time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _head_shards(rank, world, port, result):
    _init(rank, world, port)
    import oracle
    from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv
    B, S, H, D, r = 2, 96, 4, 64, 16
    qkv = make_qkv(B, S, H, D, seed=77)  # every rank draws the same full input
    per = H // world
    h0, h1 = rank * per, (rank + 1) * per
    shard = qkv[:, :, h0:h1].contiguous()
    out, lse = oracle.fwd(bf16_bits(shard), B, S, h1 - h0, D, r, 1e4, threads=1)
    outs = [torch.empty((B, S, per, D), dtype=torch.float64) for _ in range(world)]
    lses = [torch.empty((B, per, S), dtype=torch.float64) for _ in range(world)]
    dist.all_gather(outs, torch.from_numpy(out))
    dist.all_gather(lses, torch.from_numpy(lse))
    if rank == 0:
        full_out, full_lse = oracle.fwd(bf16_bits(qkv), B, S, H, D, r, 1e4, threads=1)
        got_out = torch.cat(outs, dim=2).numpy()
        got_lse = torch.cat(lses, dim=1).numpy()
        result["equal"] = bool(np.array_equal(got_out, full_out) and np.array_equal(got_lse, full_lse))
    dist.barrier()
    dist.destroy_process_group()


def _bwd_head_shards(rank, world, port, result):
    # the backward is per head too: each rank's head range, gathered, is the whole gradient
    _init(rank, world, port)
    import oracle
    from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv
    B, S, H, D, r = 1, 64, 4, 64, 16
    qkv = make_qkv(B, S, H, D, seed=78)
    dout = torch.randn((B, S, H, D), generator=torch.Generator().manual_seed(79)).to(torch.bfloat16)
    per = H // world
    h0, h1 = rank * per, (rank + 1) * per
    g = oracle.bwd(bf16_bits(qkv[:, :, h0:h1].contiguous()), bf16_bits(dout[:, :, h0:h1].contiguous()),
                   B, S, per, D, r, threads=1)
    parts = [torch.empty((B, S, per, 3, D), dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(g))
    if rank == 0:
        full = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, r, threads=1)
        result["equal"] = bool(np.array_equal(torch.cat(parts, dim=2).numpy(), full))
    dist.barrier()
    dist.destroy_process_group()


def _timing(rank, world, port, result):
    _init(rank, world, port)
    import bench
    local = [12.5, 20.0][rank]
    slowest = bench.max_over_ranks(local, dist, "cpu")
    result[f"max{rank}"] = slowest
    result[f"tflops{rank}"] = bench.job_tflops(1e12, world, 10, slowest)
    dist.barrier()
    dist.destroy_process_group()


def _spawn(fn):
    world = 2
    port = free_port()
    with mp.Manager() as m:
        result = m.dict()
        mp.spawn(fn, args=(world, port, result), nprocs=world, join=True)
        return dict(result)


def test_head_shards_gather_to_the_full_result():
    assert _spawn(_head_shards)["equal"]


def test_backward_head_shards_gather_to_the_full_gradient():
    assert _spawn(_bwd_head_shards)["equal"]


def test_benchmark_timing_is_max_over_ranks():
    r = _spawn(_timing)
    assert r["max0"] == r["max1"] == 20.0
    # two ranks x 10 steps x 1 TFLOP each in 20 ms
    assert r["tflops0"] == pytest.approx(2 * 10 * 1e12 / 0.020 / 1e12)
