"""beam_moe_route_noalloc: the router for callers that must not have the library allocate
device memory (an engine that has already claimed all free HBM, or a per-token path where
an allocator call could synchronise the device or stall). It keeps its scratch in a fixed
array inside the library instead of the stream-ordered pool, so it must give exactly what
beam_moe_route_ex gives on the same inputs.

This file is named to be collected last: if it fails, a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_moe_transformer_bias_b300 import abi, build, workloads as W

FAKE = 1 << 20  # 16-byte aligned; argument checks return before any device access


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def test_noalloc_rejects_batches_above_its_limit(lib):
    cfg = abi.BeamMoeConfig.of(W.BEAM)
    T = abi.BEAM_MOE_NOALLOC_MAX_TOKENS + 1
    rc = lib.beam_moe_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, FAKE, T, FAKE, FAKE, None)
    assert rc == abi.BEAM_MOE_ERR_ARG
    msg = abi.beam_moe_last_error()
    assert f"T={T}" in msg and str(abi.BEAM_MOE_NOALLOC_MAX_TOKENS) in msg
    assert lib.beam_moe_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, None, 4, FAKE, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert lib.beam_moe_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, FAKE, 0, FAKE, FAKE, None) == abi.BEAM_MOE_OK


def _route_regular(shape, x, wr, b):
    T = x.shape[0]
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    abi.beam_moe_route_ex(shape, x, wr, b, T, idx, w)
    return idx, w


def _route_noalloc(shape, x, wr, b):
    T = x.shape[0]
    idx = torch.full((T, shape.top_k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, shape.top_k), float("nan"), dtype=torch.float32, device="cuda")
    abi.beam_moe_route_noalloc(shape, x, wr, b, T, idx, w)
    return idx, w


@pytest.mark.gpu
@pytest.mark.parametrize("shape_name,T", [("tiny", 129), ("beam", 16), ("beam", 64), ("beam", 7040),
                                          ("beam", abi.BEAM_MOE_NOALLOC_MAX_TOKENS)])
def test_noalloc_route_matches_route_on_two_calls_in_a_row(shape_name, T):
    """Two no-allocation calls back to back on different inputs (the second reuses the
    array the first left behind), each against the regular entry point: indices bit for
    bit, weights within the routing tolerance of the other router tests (1e-6 relative).
    T=16 runs the small-batch router, the others the tensor-core one; T=7040 is the batch
    whose router scratch fills the most of the array on a 148-SM B300."""
    shape = W.TINY if shape_name == "tiny" else W.BEAM
    inputs = []
    for seed in (0, 1):
        x = W.make_tokens(shape, T, seed, "cuda")
        wr, b = W.make_router(shape, seed, "cuda")
        inputs.append((x, wr, b))
    got = [_route_noalloc(shape, *inp) for inp in inputs]   # two calls in a row, one stream
    want = [_route_regular(shape, *inp) for inp in inputs]
    torch.cuda.synchronize()
    abi.beam_moe_device_status()
    for (gi, gw), (wi, ww) in zip(got, want):
        gi, gw, wi, ww = (t.cpu().numpy() for t in (gi, gw, wi, ww))
        np.testing.assert_array_equal(gi, wi)
        np.testing.assert_allclose(gw, ww, rtol=1e-6, atol=1e-7)
        assert np.all(np.abs(gw.sum(axis=1) - shape.scale) <= 1e-5)
    assert not np.array_equal(got[0][0].cpu().numpy(), got[1][0].cpu().numpy())
