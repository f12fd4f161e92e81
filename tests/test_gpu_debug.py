"""The scratch-poison debug aid: with every scratch allocation filled with NaN bytes
before use, each entry point must give bit for bit what it gives without it. A kernel
that read a scratch value it had not written (a row of x_perm, h or y, a partial logit
plane, a work-list entry) would turn that NaN or -1 into a changed output or a recorded
index error."""
import pytest
import torch

from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def _both(fn):
    """fn() without and with the poison; both results and a clean status word."""
    abi.beam_moe_debug_poison_scratch(False)
    a = fn()
    torch.cuda.synchronize()
    abi.beam_moe_debug_poison_scratch(True)
    try:
        b = fn()
        torch.cuda.synchronize()
    finally:
        abi.beam_moe_debug_poison_scratch(False)
    abi.beam_moe_device_status()
    return a, b


def _tiny(T, seed=0, shape=W.TINY):
    x = W.make_tokens(shape, T, seed, "cuda")
    wr, b = W.make_router(shape, seed, "cuda")
    return shape, x, wr, b, W.make_experts(shape, seed, "cuda")


@pytest.mark.parametrize("T", [1, 7, 129, 300])
def test_forward_unchanged_by_poisoned_scratch(T):
    shape, x, wr, b, (wg, wu, wd) = _tiny(T)
    a, p = _both(lambda: moe.forward(x, wr, b, wg, wu, wd, shape))
    assert not torch.isnan(p.float()).any()
    assert torch.equal(a, p)
    ra, rp = _both(lambda: moe.route(x, wr, b, shape))
    assert all(torch.equal(u, v) for u, v in zip(ra, rp))


def test_beam_decode_and_prefill_sized_calls_unchanged(beam_experts):
    shape = W.BEAM
    for T in (16, 1024):
        x = W.make_tokens(shape, T, 0, "cuda")
        wr, b = W.make_router(shape, 0, "cuda")
        a, p = _both(lambda: moe.forward(x, wr, b, *beam_experts, shape))
        assert torch.equal(a, p), T


def test_other_entry_points_unchanged():
    shape, x, wr, b, (wg, wu, wd) = _tiny(300, seed=1)
    a, p = _both(lambda: moe.forward_shard(x, wr, b, wg[64:128].contiguous(), wu[64:128].contiguous(),
                                           wd[64:128].contiguous(), 64, 128, shape))
    assert torch.equal(a, p)
    q = W.make_experts_fp8(shape, 1, "cuda")
    a, p = _both(lambda: moe.forward_fp8(x, wr, b, q, shape))
    assert torch.equal(a, p)
    g = torch.ones(shape.d, dtype=torch.bfloat16, device="cuda")
    a, p = _both(lambda: moe.sublayer_forward(x, g, g, 1e-6, 5, wr, b, wg, wu, wd, shape))
    assert torch.equal(a, p)
    a, p = _both(lambda: moe.dense_mlp(x, wg[0], wu[0], wd[0]))
    assert torch.equal(a, p)


@pytest.mark.parametrize("T", [7, 300])
def test_nvfp4_unchanged_by_poisoned_scratch(T):
    """The NVFP4 block keeps its activation pieces, their scales and h's pieces in scratch;
    piece rows past a tile's tokens (read as padding of the products) may hold the poison,
    which must stay out of every stored value and out of the range check."""
    shape = W.TINY
    x = W.make_tokens(shape, T, 2, "cuda")
    wr, b = W.make_router(shape, 2, "cuda")
    q4 = W.make_experts_nvfp4(shape, 2, "cuda")
    a, p = _both(lambda: moe.forward_nvfp4(x, wr, b, q4, shape))
    assert not torch.isnan(p.float()).any()
    assert torch.equal(a, p)
