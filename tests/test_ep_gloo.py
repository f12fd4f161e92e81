"""Multi-process paths on the CPU (gloo, world size 2, no GPU).

Expert parallelism as the pages deploy it (each expert on one device, the rest replicated;
Glonce "Reflection releases Beam ...", Running it paragraph): rank r owns a contiguous half of
the experts, computes its shard's partial output with the oracle, and the partials meet in an
all-reduce sum, which must equal the whole block. The benchmark's barrier and max-over-ranks
timing are exercised the same way."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_moe_transformer_bias_b300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ep_worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle as O
        shape = W.MoEShape(d=128, I=128, E=64, n_group=2, topk_group=1, top_k=8)
        T = 20
        x = W.make_tokens(shape, T, 3)
        wr, b = W.make_router(shape, 3)
        wg, wu, wd = W.make_experts(shape, 3)
        xb = O.bf16_bits(x)
        per = shape.E // world
        lo, hi = rank * per, (rank + 1) * per
        experts = O.experts_from(wg, wu, wd)
        part = O.forward_shard(shape, xb, b.numpy(), experts, lo, hi, np.arange(T), router_w=wr.numpy())
        t = torch.from_numpy(part)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            full, _, _ = O.forward(shape, xb, b.numpy(), experts, router_w=wr.numpy())
            results["max_err"] = float(np.abs(t.numpy() - full).max())
            results["scale"] = float(np.abs(full).max())
        import bench
        bench.barrier()
        results[f"max_{rank}"] = bench.max_over_ranks(10.0 + rank)
    finally:
        dist.destroy_process_group()


def test_expert_parallel_shards_sum_to_the_block_over_gloo():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (possibly CUDA) process
        results = m.dict()
        mp.spawn(_ep_worker, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res["max_err"] <= 1e-12 * max(1.0, res["scale"]), res
    assert res["max_0"] == res["max_1"] == 11.0
