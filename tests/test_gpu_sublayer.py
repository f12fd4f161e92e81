"""The MoE sublayer on the residual stream (pre-RMSNorm, MoE block, post-RMSNorm fused with
the depth-scaled residual) and the standalone RMSNorm: CUDA library against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import parity as P
from oracle import oracle as O
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu

EPS = 1e-6


def norm_inputs(shape, T, seed, scale=3.0):
    g = torch.Generator(device="cuda").manual_seed(1000 + seed)
    stream = (torch.randn((T, shape.d), generator=g, device="cuda") * scale).to(torch.bfloat16)
    pre = (1.0 + 0.1 * torch.randn(shape.d, generator=g, device="cuda")).to(torch.bfloat16)
    post = (1.0 + 0.1 * torch.randn(shape.d, generator=g, device="cuda")).to(torch.bfloat16)
    return stream, pre, post


def check_norm_rows(gpu_bits_rows, ref_rows, what):
    """BF16 output of an FP32 RMSNorm against the FP64 oracle: within one BF16 step
    (2^-8 relative) of the exact value."""
    g = (gpu_bits_rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(g - ref_rows)
    bound = 2.0 ** -8 * np.abs(ref_rows) + 1e-30
    assert np.all(err <= bound), f"{what}: max rel err {np.max(err / (np.abs(ref_rows) + 1e-30))}"


@pytest.mark.parametrize("d,T", [(512, 1), (512, 37), (5120, 16), (5120, 300), (8192, 5), (4, 3)])
def test_rmsnorm_parity(d, T):
    shape = W.MoEShape(d=d, I=256)
    stream, pre, _ = norm_inputs(shape, T, seed=d + T)
    out = moe.rmsnorm(stream, pre, EPS)
    torch.cuda.synchronize()
    sb = O.bf16_bits(stream)
    ref = np.stack([O.rmsnorm((sb[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64),
                              O.bf16_bits(pre), EPS) for t in range(T)])
    check_norm_rows(O.bf16_bits(out), ref, f"rmsnorm d={d} T={T}")


def test_rmsnorm_in_place_and_deterministic():
    shape = W.TINY
    stream, pre, _ = norm_inputs(shape, 50, seed=3)
    a = moe.rmsnorm(stream, pre, EPS)
    b = stream.clone()
    moe.rmsnorm(b, pre, EPS, out=b)
    c = moe.rmsnorm(stream, pre, EPS)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def run_sublayer(layer, stream, pre, post, k):
    shape = layer.shape
    out = moe.sublayer_forward(stream, pre, post, EPS, k, layer.wr, layer.b, layer.wg, layer.wu, layer.wd, shape)
    x = moe.rmsnorm(stream, pre, EPS)
    logits = moe.router_logits(x, layer.wr, shape)
    idx, _ = moe.route(x, layer.wr, layer.b, shape)
    abi.beam_moe_device_status()
    return out, x, logits.cpu().numpy(), idx.cpu().numpy()


def check_sublayer(layer, stream, pre, post, k, tokens, what):
    out, x, logits, idx = run_sublayer(layer, stream, pre, post, k)
    tokens = np.asarray(tokens, np.int64)
    shape = layer.shape
    xb = O.bf16_bits(x)
    # the GPU's pre-norm, against the oracle's (one BF16 step)
    s_rows = (O.bf16_bits(stream)[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x_ref = np.stack([O.rmsnorm(s_rows[i], O.bf16_bits(pre), EPS) for i in range(len(tokens))])
    check_norm_rows(xb[tokens], x_ref, f"{what} pre-norm")
    # the rest of the sublayer given the GPU's BF16 input and FP32 logits
    _, _, dbg = O.route(shape, logits[tokens], layer.b.cpu().numpy(), debug=True)
    flagged = P.near_tie_tokens(shape, dbg)
    needed = set(np.unique(idx[tokens]).tolist())
    idx_r, _ = O.route(shape, logits[tokens], layer.b.cpu().numpy())
    needed |= set(np.unique(idx_r).tolist())
    experts = layer.experts(needed)
    grouped = len(tokens) > 64
    ref, _ = O.sublayer(shape, O.bf16_bits(stream), O.bf16_bits(pre), O.bf16_bits(post), EPS, k,
                        layer.b.cpu().numpy(), experts, tokens, x_bits=xb, logits=logits, grouped=grouped)
    if len(flagged):
        ref2, _ = O.sublayer(shape, O.bf16_bits(stream), O.bf16_bits(pre), O.bf16_bits(post), EPS, k,
                             layer.b.cpu().numpy(), experts, tokens[flagged], x_bits=xb, logits=logits,
                             idx_in=idx[tokens[flagged]], grouped=grouped)
        ref[flagged] = ref2
    got = out.float().cpu().numpy()[tokens]
    frob = P.check_output(got, ref, what)
    print(f"{what}: tokens {len(tokens)}, near-tie {len(flagged)}, rel frob {frob:.2e}")
    return out


@pytest.mark.parametrize("T,k", [(7, 2), (129, 7), (300, 105)])
def test_tiny_sublayer_parity(T, k):
    shape = W.TINY
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    wg, wu, wd = W.make_experts(shape, 0, "cuda")
    layer = P.Layer(shape, x, wr, b, wg, wu, wd)
    stream, pre, post = norm_inputs(shape, T, seed=T)
    check_sublayer(layer, stream, pre, post, k, np.arange(T), f"tiny sublayer T={T} k={k}")


@pytest.mark.parametrize("T,k,n_check", [(16, 9, 16), (1024, 53, 256)])
def test_beam_sublayer_parity(beam_experts, beam_host_cache, T, k, n_check):
    shape = W.BEAM
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    layer = P.Layer(shape, x, wr, b, *beam_experts, host_cache=beam_host_cache)
    stream, pre, post = norm_inputs(shape, T, seed=T)
    tokens = np.unique(np.concatenate([W.sample_tokens(T, n_check, seed=5).numpy(), [T - 1]]))
    check_sublayer(layer, stream, pre, post, k, tokens, f"beam sublayer T={T} k={k}")


def test_zero_post_gain_keeps_the_scaled_stream():
    """post_gamma = 0: the sublayer contributes nothing, so the stream is only rescaled by
    sqrt((k-1)/k) (one FP32 multiply, rounded once to BF16): bit-exact."""
    shape = W.TINY
    T, k = 64, 11
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    wg, wu, wd = W.make_experts(shape, 0, "cuda")
    stream, pre, _ = norm_inputs(shape, T, seed=9)
    post = torch.zeros(shape.d, dtype=torch.bfloat16, device="cuda")
    out = moe.sublayer_forward(stream, pre, post, EPS, k, wr, b, wg, wu, wd, shape)
    a = torch.tensor(math.sqrt((k - 1) / k), dtype=torch.float32)
    want = (stream.float().cpu() * a).to(torch.bfloat16)
    assert torch.equal(out.cpu(), want)


def test_sublayer_in_place_and_deterministic():
    shape = W.TINY
    T, k = 129, 5
    wr, b = W.make_router(shape, 2, "cuda")
    wg, wu, wd = W.make_experts(shape, 2, "cuda")
    stream, pre, post = norm_inputs(shape, T, seed=4)
    a = moe.sublayer_forward(stream, pre, post, EPS, k, wr, b, wg, wu, wd, shape)
    c = moe.sublayer_forward(stream, pre, post, EPS, k, wr, b, wg, wu, wd, shape)
    s2 = stream.clone()
    moe.sublayer_forward(s2, pre, post, EPS, k, wr, b, wg, wu, wd, shape, out=s2)
    torch.cuda.synchronize()
    assert torch.equal(a, c) and torch.equal(a, s2)
    assert abi.beam_moe_last_launch_count() == len(abi.STAGES) - 1  # every stage but the FP8 prep


def test_sublayer_keeps_the_stream_scale():
    """The pages' point of the depth scaling: with a unit-RMS stream and unit post-gain,
    the updated stream stays near unit RMS (the normalised sublayer output has unit RMS and
    is nearly uncorrelated with the stream)."""
    shape = W.TINY
    T, k = 256, 9
    wr, b = W.make_router(shape, 1, "cuda")
    wg, wu, wd = W.make_experts(shape, 1, "cuda")
    stream, pre, _ = norm_inputs(shape, T, seed=8, scale=1.0)
    post = torch.ones(shape.d, dtype=torch.bfloat16, device="cuda")
    out = moe.sublayer_forward(stream, pre, post, EPS, k, wr, b, wg, wu, wd, shape).float()
    rms = out.pow(2).mean(dim=1).sqrt()
    assert float((rms - 1.0).abs().max()) < 0.1
