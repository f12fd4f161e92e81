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


def _splits_unconstrained(shape, T, num_sms):
    """The K split count the regular router picks (its cost model restated: per item ~550 ns
    per 64-wide K chunk plus ~1500 ns, in waves over the SMs, plus the partial planes at
    ~6 TB/s; ties to fewer splits); 1 on the CUDA-core path for T <= 32."""
    if T <= 32:
        return 1
    kc = shape.d // 64
    tiles = -(-T // 128) * -(-shape.E // 128)
    best, best_cost = 1, None
    for sp in range(1, min(16, kc) + 1):
        if kc % sp:
            continue
        waves = -(-(tiles * sp) // num_sms)
        cost = waves * ((kc // sp) * 550 + 1500) + sp * T * shape.E * 8 // 6000
        if best_cost is None or cost < best_cost:
            best, best_cost = sp, cost
    return best


def _fits(shape, T, sp):
    w3 = 0 if T <= 32 else (3 * shape.E * shape.d * 2 + 255) // 256 * 256
    return w3 + sp * T * shape.E * 4 <= abi.BEAM_MOE_NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("num_sms", [148, 160, 170, 192])
def test_noalloc_plan_fits_the_array(lib, num_sms):
    """The planning query (host only): its split count divides the d/64 K chunks, fits the
    fixed array, equals the regular router's choice whenever that fits (always on a 148-SM
    B300 up to the token limit) and is otherwise the largest dividing count below it that
    fits. More SMs make the regular router pick more splits: up to 170 SMs every choice
    still fits, at 192 the larger batches run the reduction."""
    shape = W.BEAM
    reduced = 0
    for T in list(range(1, 65)) + list(range(96, abi.BEAM_MOE_NOALLOC_MAX_TOKENS + 1, 160)) + [7040, 8191, 8192]:
        sp = abi.beam_moe_route_noalloc_plan(shape, T, num_sms)
        want = _splits_unconstrained(shape, T, num_sms)
        kc = shape.d // 64
        assert kc % sp == 0 and _fits(shape, T, sp), (T, sp)
        if _fits(shape, T, want):
            assert sp == want, (T, sp, want)
        else:
            reduced += 1
            assert sp < want and not any(_fits(shape, T, c) for c in range(sp + 1, want + 1) if kc % c == 0), (T, sp)
    assert (reduced == 0) == (num_sms <= 170), (num_sms, reduced)


def test_noalloc_plan_rejects_what_does_not_fit(lib):
    cfg = abi.BeamMoeConfig.of(W.BEAM)
    n = ctypes.c_int(-1)
    for T in (0, -3, abi.BEAM_MOE_NOALLOC_MAX_TOKENS + 1):
        assert lib.beam_moe_route_noalloc_plan(ctypes.byref(cfg), T, 148, ctypes.byref(n)) == abi.BEAM_MOE_ERR_ARG
    assert lib.beam_moe_route_noalloc_plan(ctypes.byref(cfg), 64, 0, ctypes.byref(n)) == abi.BEAM_MOE_ERR_ARG
    assert lib.beam_moe_route_noalloc_plan(ctypes.byref(cfg), 64, 148, None) == abi.BEAM_MOE_ERR_ARG
    # router weight pieces of 3 * 256 * 32768 BF16 (48 MiB) alone exceed the 40 MiB array
    wide = abi.BeamMoeConfig(32768, 2560, 256, 8, 4, 8, 2.5)
    assert lib.beam_moe_route_noalloc_plan(ctypes.byref(wide), 64, 148, ctypes.byref(n)) == abi.BEAM_MOE_ERR_ARG
    assert "more router scratch" in abi.beam_moe_last_error()
    assert n.value == -1


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
    abi.beam_moe_route_noalloc_status()
    for (gi, gw), (wi, ww) in zip(got, want):
        gi, gw, wi, ww = (t.cpu().numpy() for t in (gi, gw, wi, ww))
        np.testing.assert_array_equal(gi, wi)
        np.testing.assert_allclose(gw, ww, rtol=1e-6, atol=1e-7)
        assert np.all(np.abs(gw.sum(axis=1) - shape.scale) <= 1e-5)
    assert not np.array_equal(got[0][0].cpu().numpy(), got[1][0].cpu().numpy())


@pytest.mark.gpu
def test_noalloc_route_allocates_no_device_memory():
    """The property the entry point exists for, in a fresh process (where the library's
    pool has never been created): after one warm-up call (the array is part of the loaded
    device image, and the first call looks up its address), more calls at the token limit
    leave the device's free memory unchanged, and the library's regular pool is never
    created."""
    import subprocess
    import sys
    code = r"""
import torch
from sparse_moe_transformer_bias_b300 import abi, workloads as W
shape, T = W.BEAM, abi.BEAM_MOE_NOALLOC_MAX_TOKENS
x = W.make_tokens(shape, T, 0, "cuda")
wr, b = W.make_router(shape, 0, "cuda")
idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
w = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
abi.beam_moe_route_noalloc(shape, x, wr, b, T, idx, w)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    abi.beam_moe_route_noalloc(shape, x, wr, b, T, idx, w)
    abi.beam_moe_route_noalloc(shape, x[:16], wr, b, 16, idx, w)
torch.cuda.synchronize()
abi.beam_moe_route_noalloc_status()
free1 = torch.cuda.mem_get_info()[0]
print("FREE", free0, free1)
"""
    root = __import__("os").path.dirname(__import__("os").path.dirname(__import__("os").path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1]
    free0, free1 = (int(v) for v in line.split()[1:])
    assert free1 == free0, (free0, free1)


@pytest.mark.gpu
def test_noalloc_wait_timeout_is_reported_on_its_own_status_word():
    """Failure detection of the no-allocation router without a GPU fault: the self-test makes
    one bounded wait of its logits kernel run out (2 s); beam_moe_route_noalloc_status
    reports it once and clears it, the library's other status word stays clean, and the
    same context then routes exactly as before."""
    shape, T = W.BEAM, 64
    x = W.make_tokens(shape, T, 3, "cuda")
    wr, b = W.make_router(shape, 3, "cuda")
    before = _route_noalloc(shape, x, wr, b)
    abi.beam_moe_route_noalloc_status()
    abi.beam_moe_route_noalloc_selftest()
    with pytest.raises(abi.BeamMoeError) as err:
        abi.beam_moe_route_noalloc_status()
    assert err.value.code == abi.BEAM_MOE_ERR_DEVICE and "ran past its limit" in str(err.value)
    abi.beam_moe_route_noalloc_status()  # cleared by the read
    abi.beam_moe_device_status()         # the regular entry points' word was not touched
    after = _route_noalloc(shape, x, wr, b)
    abi.beam_moe_route_noalloc_status()
    for a, c in zip(before, after):
        assert torch.equal(a, c)
