"""The forward pass captured in a CUDA graph and replayed gives the direct call's result
bit for bit, also after new tokens are written into the captured input buffer."""
import pytest
import torch

from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape_name,T", [("tiny", 16), ("tiny", 300), ("beam", 16)])
def test_graph_replay_matches_direct_call(shape_name, T, beam_experts):
    shape = W.TINY if shape_name == "tiny" else W.BEAM
    wr, b = W.make_router(shape, 3, "cuda")
    experts = W.make_experts(shape, 3, "cuda") if shape_name == "tiny" else beam_experts
    x = W.make_tokens(shape, T, 3, "cuda")
    g = moe.ForwardGraph(x, wr, b, *experts, shape)
    got = g.replay().clone()
    want = moe.forward(x, wr, b, *experts, shape)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    x2 = W.make_tokens(shape, T, 4, "cuda")
    g.x.copy_(x2)
    got2 = g.replay().clone()
    want2 = moe.forward(x2, wr, b, *experts, shape)
    abi.beam_moe_device_status()
    assert torch.equal(got2, want2)
    assert not torch.equal(got, got2)
