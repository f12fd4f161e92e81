"""Expert parallelism across processes: two ranks, each a separate process holding half of
the experts (the pages' plan: each expert on one device, the rest replicated; Glonce
"Reflection releases Beam ...", Running it paragraph; transformers "Beam" doc, Usage
examples: expert parallelism under torchrun). Each rank runs beam_moe_forward_shard through
the C ABI on its own experts; the FP32 partials meet in an all-reduce sum over gloo (host
copies: every run here has one GPU, so both ranks share it; their kernels never wait on
each other). The sum must equal the unsharded block within one BF16 step and the oracle
within the output tolerance."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import parity as P
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape(name):
    return W.TINY if name == "tiny" else W.BEAM


def _rank_worker(rank, world, port, name, T, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        shape = _shape(name)
        x = W.make_tokens(shape, T, 0, "cuda")
        wr, b = W.make_router(shape, 0, "cuda")
        per = shape.E // world
        lo, hi = rank * per, (rank + 1) * per
        wg, wu, wd = (w[lo:hi].contiguous() for w in W.make_experts(shape, 0, "cuda"))
        torch.cuda.empty_cache()
        part = moe.forward_shard(x, wr, b, wg, wu, wd, lo, hi, shape)
        abi.beam_moe_device_status()
        t = part.cpu()
        results[f"own_{rank}"] = t.numpy().copy()
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            results["sum"] = t.numpy().copy()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,T", [("tiny", 129), ("beam", 16)])
def test_two_process_expert_parallel_shards_sum_to_the_block(beam_experts, beam_host_cache, name, T):
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (possibly CUDA) process
        results = m.dict()
        mp.spawn(_rank_worker, args=(2, port, name, T, results), nprocs=2, join=True)
        res = dict(results)
    total = torch.from_numpy(res["sum"])
    assert np.array_equal(res["own_0"] + res["own_1"], res["sum"])  # the all-reduce is that sum
    shape = _shape(name)
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    experts = beam_experts if name == "beam" else W.make_experts(shape, 0, "cuda")
    out = moe.forward(x, wr, b, *experts, shape).float().cpu()
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    idx, _ = moe.route(x, wr, b, shape)
    abi.beam_moe_device_status()
    # the unsharded call: the same slot sum in another FP32 order, rounded to BF16
    diff = (total.to(torch.bfloat16).float() - out).abs()
    assert float((diff - 2.0 ** -7 * out.abs()).max()) <= 1e-6
    layer = P.Layer(shape, x, wr, b, *experts, host_cache=beam_host_cache if name == "beam" else {})
    ref, flagged = P.oracle_forward_for(layer, np.arange(T), logits, idx.cpu().numpy())
    frob = P.check_output(total.numpy(), ref, f"{name} 2 processes")
    print(f"{name} T={T} 2 processes: rel frob {frob:.2e}, near-tie {len(flagged)}")
