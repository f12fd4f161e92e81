"""Expert-parallel shards on one GPU: every shard computes its partial output through the C
ABI with only its experts' weights; the shards, run one after another, must add up to the
unsharded block (expert-parallel plan: each expert on one device, the combine a sum over
devices; Glonce "Reflection releases Beam ...", Running it paragraph)."""
import numpy as np
import pytest
import torch

import parity as P
from oracle import oracle as O
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def shard_sum(layer, n_shards):
    shape = layer.shape
    per = shape.E // n_shards
    total = torch.zeros((layer.x.shape[0], shape.d), dtype=torch.float32, device="cuda")
    parts = []
    for r in range(n_shards):
        lo, hi = r * per, (r + 1) * per
        part = moe.forward_shard(layer.x, layer.wr, layer.b, layer.wg[lo:hi].contiguous(),
                                 layer.wu[lo:hi].contiguous(), layer.wd[lo:hi].contiguous(), lo, hi, shape)
        parts.append(part)
        total += part
    abi.beam_moe_device_status()
    return total, parts


def tiny_layer(T, seed=0):
    shape = W.TINY
    x = W.make_tokens(shape, T, seed, "cuda")
    wr, b = W.make_router(shape, seed, "cuda")
    wg, wu, wd = W.make_experts(shape, seed, "cuda")
    return P.Layer(shape, x, wr, b, wg, wu, wd)


@pytest.mark.parametrize("n_shards", [2, 4, 8])
def test_tiny_shards_add_up_to_the_block(n_shards):
    layer = tiny_layer(129)
    total, parts = shard_sum(layer, n_shards)
    out = moe.forward(layer.x, layer.wr, layer.b, layer.wg, layer.wu, layer.wd, layer.shape)
    logits = moe.router_logits(layer.x, layer.wr, layer.shape).cpu().numpy()
    idx, _ = moe.route(layer.x, layer.wr, layer.b, layer.shape)
    torch.cuda.synchronize()
    # against the oracle (all tokens), with the usual output tolerance
    ref, flagged = P.oracle_forward_for(layer, np.arange(129), logits, idx.cpu().numpy())
    frob = P.check_output(total.cpu().numpy(), ref, f"tiny {n_shards} shards")
    # against the unsharded call: the same sum in another FP32 order, rounded to BF16
    diff = (total.to(torch.bfloat16).float() - out.float()).abs()
    assert float((diff - 2.0 ** -7 * out.float().abs()).max()) <= 1e-6
    print(f"tiny {n_shards} shards: rel frob {frob:.2e}, near-tie {len(flagged)}")


def test_tiny_shard_partial_against_oracle():
    """One shard's partial alone (experts 64..127 of 256), every token, against the oracle's
    sum over the token's slots routed there."""
    layer = tiny_layer(40, seed=3)
    shape = layer.shape
    lo, hi = 64, 128
    part = moe.forward_shard(layer.x, layer.wr, layer.b, layer.wg[lo:hi].contiguous(), layer.wu[lo:hi].contiguous(),
                             layer.wd[lo:hi].contiguous(), lo, hi, shape)
    logits = moe.router_logits(layer.x, layer.wr, shape).cpu().numpy()
    abi.beam_moe_device_status()
    _, _, dbg = O.route(shape, logits, layer.b.cpu().numpy(), debug=True)
    assert len(P.near_tie_tokens(shape, dbg)) == 0
    experts = layer.experts(set(range(lo, hi)))
    ref = O.forward_shard(shape, O.bf16_bits(layer.x), layer.b.cpu().numpy(), experts, lo, hi, np.arange(40),
                          logits=logits)
    got = part.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 2e-2 * np.abs(ref))
    assert np.linalg.norm(got - ref) <= 5e-3 * max(np.linalg.norm(ref), 1e-30)
    # tokens with no slot on the shard read exactly 0
    idx_o, _ = O.route(shape, logits, layer.b.cpu().numpy())
    none_here = ~((idx_o >= lo) & (idx_o < hi)).any(axis=1)
    assert np.all(got[none_here] == 0.0)


@pytest.mark.parametrize("name,T,n_check", [("decode", 16, 16), ("prefill", 4096, 24)])
def test_beam_eight_shards_add_up_to_the_block(beam_experts, beam_host_cache, name, T, n_check):
    """Beam shapes, 8 shards of 32 experts (the pages' 8-device plan), emulated one after
    another on one GPU."""
    shape = W.BEAM
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    layer = P.Layer(shape, x, wr, b, *beam_experts, host_cache=beam_host_cache)
    total, _ = shard_sum(layer, 8)
    out = moe.forward(x, wr, b, *beam_experts, shape)
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    idx, _ = moe.route(x, wr, b, shape)
    torch.cuda.synchronize()
    tokens = W.sample_tokens(T, n_check, seed=2).numpy()
    ref, _ = P.oracle_forward_for(layer, tokens, logits, idx.cpu().numpy())
    frob = P.check_output(total.cpu().numpy()[tokens], ref, f"{name} 8 shards")
    diff = (total.to(torch.bfloat16).float() - out.float()).abs()
    assert float((diff - 2.0 ** -7 * out.float().abs()).max()) <= 1e-6
    print(f"{name} 8 shards: rel frob {frob:.2e}")
