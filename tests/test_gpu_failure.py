"""Failure detection on the GPU without a fault: the library's self-test makes one bounded
wait of the expert kernel run out (its completion counter can never reach the count the
down item waits for). The kernel must record the timeout in the status word, leave its
pipeline in order and return; the host reads the code, the word is cleared, and the same
context keeps producing the same results."""
import pytest
import torch

from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def tiny_forward(T=33, seed=12):
    shape = W.TINY
    x = W.make_tokens(shape, T, seed, "cuda")
    wr, b = W.make_router(shape, seed, "cuda")
    wg, wu, wd = W.make_experts(shape, seed, "cuda")
    return lambda: moe.forward(x, wr, b, wg, wu, wd, shape)


def test_wait_timeout_is_reported_and_the_context_survives():
    run = tiny_forward()
    assert abi.beam_moe_device_status() == abi.BEAM_MOE_OK
    before = run()
    torch.cuda.synchronize()
    abi.beam_moe_selftest_wait_timeout()
    with pytest.raises(abi.BeamMoeError, match="ran past its limit") as err:
        abi.beam_moe_device_status()
    assert err.value.code == abi.BEAM_MOE_ERR_DEVICE
    assert abi.beam_moe_device_status() == abi.BEAM_MOE_OK  # the word was cleared
    after = run()
    abi.beam_moe_device_status()
    assert torch.equal(before, after)
