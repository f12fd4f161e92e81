"""FP8 expert weights: the CUDA block with E4M3 codes and per-row FP32 scales against the
oracle on the same codes and scales (forward_fp8), element by element, on Tiny (every
token, ragged counts, both N-tile sizes of the FP8 kernel) and on Beam shapes (sampled
tokens at full size), plus a case that puts every finite E4M3 code through the widening."""
import numpy as np
import pytest
import torch

import parity as P
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def host_experts(q8, cache=None):
    """Oracle callable e -> (wg_q, gs, wu_q, us, wd_q, ds) over device FP8 experts, copying
    an expert to the host on first use."""
    (wg, gs), (wu, us), (wd, ds) = q8
    cache = {} if cache is None else cache

    def get(e):
        if e not in cache:
            cache[e] = tuple(t[e].cpu().numpy() for t in (wg, gs, wu, us, wd, ds))
        return cache[e]
    return get


def run_and_check(shape, x, wr, b, q8, tokens, what, cache=None):
    out = moe.forward_fp8(x, wr, b, q8, shape)
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    idx, _ = moe.route(x, wr, b, shape)
    abi.beam_moe_device_status()
    out = out.float().cpu().numpy()
    ref, flagged = P.oracle_forward_fp8_for(shape, x, b, host_experts(q8, cache), tokens, logits, idx.cpu().numpy())
    frob = P.check_output(out[np.asarray(tokens)], ref, what)
    print(f"{what}: tokens checked {len(tokens)}, near-tie {len(flagged)}, rel frob {frob:.2e}")
    return out


@pytest.fixture(scope="module")
def tiny_fp8():
    return W.make_experts_fp8(W.TINY, seed=0, device="cuda")


@pytest.mark.parametrize("T", [1, 16, 33, 129, 300, 1500])
def test_tiny_fp8_parity(tiny_fp8, T):
    shape = W.TINY
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    run_and_check(shape, x, wr, b, tiny_fp8, np.arange(T), f"tiny fp8 T={T}")


def test_every_finite_code_is_widened_exactly():
    """Gate, up and down codes cycle through all 254 finite E4M3 codes (zeros, subnormals,
    both signs, +-448) in every row, scales spread over several binades: the output must
    still match the oracle on every token."""
    shape = W.TINY
    E, d, I = shape.E, shape.d, shape.I
    finite = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    gen = torch.Generator().manual_seed(11)

    def codes(rows, cols):
        out = torch.empty((E, rows, cols), dtype=torch.uint8)
        for e in range(E):
            perm = finite[torch.randperm(len(finite), generator=gen)]
            reps = (rows * cols + len(perm) - 1) // len(perm)
            out[e] = perm.repeat(reps)[: rows * cols].view(rows, cols)
        return out.cuda()

    def scales(rows, fan_in):
        s = torch.exp2(torch.randint(-3, 4, (E, rows), generator=gen).float())
        return (s / (448.0 * fan_in ** 0.5)).cuda()

    q8 = ((codes(I, d), scales(I, d)), (codes(I, d), scales(I, d)), (codes(d, I), scales(d, I)))
    T = 64
    x = W.make_tokens(shape, T, 4, "cuda")
    wr, b = W.make_router(shape, 4, "cuda")
    run_and_check(shape, x, wr, b, q8, np.arange(T), "all codes")


def test_subnormal_codes_only():
    """Weights made of the 16 codes with exponent field 0 (zeros and subnormals, both signs),
    scaled so that the outputs are O(1): a path that flushed subnormal weights, or their
    products, would lose the whole signal and fail the relative error bound."""
    shape = W.TINY
    E, d, I = shape.E, shape.d, shape.I
    pool = torch.tensor([s | m for s in (0, 0x80) for m in range(8)], dtype=torch.uint8)
    gen = torch.Generator().manual_seed(5)

    def codes(rows, cols):
        return pool[torch.randint(0, len(pool), (E, rows, cols), generator=gen)].cuda()

    def scales(rows, fan_in):
        return torch.full((E, rows), 1.0 / (0.007 * fan_in ** 0.5), device="cuda")

    q8 = ((codes(I, d), scales(I, d)), (codes(I, d), scales(I, d)), (codes(d, I), scales(d, I)))
    T = 48
    x = W.make_tokens(shape, T, 6, "cuda")
    wr, b = W.make_router(shape, 6, "cuda")
    out = run_and_check(shape, x, wr, b, q8, np.arange(T), "subnormal codes")
    assert np.abs(out).max() > 0.05


def test_fp8_deterministic(tiny_fp8):
    shape = W.TINY
    x = W.make_tokens(shape, 300, 7, "cuda")
    wr, b = W.make_router(shape, 7, "cuda")
    a = moe.forward_fp8(x, wr, b, tiny_fp8, shape)
    c = moe.forward_fp8(x, wr, b, tiny_fp8, shape)
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_fp8_close_to_bf16_block(tiny_fp8):
    """Same draws as the BF16 experts, quantised: the two blocks differ only by the
    quantisation error (about 2^-4 relative per weight, averaging out over the sums)."""
    shape = W.TINY
    x = W.make_tokens(shape, 200, 1, "cuda")
    wr, b = W.make_router(shape, 1, "cuda")
    wg, wu, wd = W.make_experts(shape, 0, "cuda")
    ref = moe.forward(x, wr, b, wg, wu, wd, shape).double()
    got = moe.forward_fp8(x, wr, b, tiny_fp8, shape).double()
    rel = float((got - ref).norm() / ref.norm())
    assert rel < 0.1, rel


@pytest.fixture(scope="module")
def beam_fp8():
    return W.make_experts_fp8(W.BEAM, seed=0, device="cuda")


@pytest.mark.parametrize("name,T,n_check", [("decode", 16, 16), ("sweep_T64", 64, 12), ("prefill", 4096, 20)])
def test_beam_fp8_parity(beam_fp8, name, T, n_check):
    shape = W.BEAM
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    tokens = W.sample_tokens(T, n_check, seed=2).numpy()
    if T > n_check:
        tokens = np.unique(np.concatenate([tokens, [T - 1]]))
    run_and_check(shape, x, wr, b, beam_fp8, tokens, f"{name} fp8 T={T}")
