"""FP8 expert weights: the CUDA block with E4M3 codes and per-row FP32 scales against the
oracle on the same codes and scales (forward_fp8), element by element, on Tiny (every
token, ragged counts, every N-tile size of the FP8 kernel: 32 rows for T <= 32, 64 and
128) and on Beam shapes (sampled tokens at full size), plus cases that put every finite
E4M3 code through the FP8 tensor cores and that stretch the on-chip split of the BF16
activations into two E4M3 pieces."""
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


@pytest.mark.parametrize("T", [1, 16, 33, 129, 300, 1500, 2100])
def test_tiny_fp8_parity(tiny_fp8, T):
    shape = W.TINY
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    run_and_check(shape, x, wr, b, tiny_fp8, np.arange(T), f"tiny fp8 T={T}")


def test_every_finite_code_is_multiplied_exactly():
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


def test_activation_rows_with_a_wide_range():
    """The on-chip split of each BF16 token row into two E4M3 pieces under one power-of-two
    row scale: rows whose largest entry is 2^12 times their typical entry (their small
    entries then fall into the E4M3 subnormal range of the pieces), rows of one tiny
    magnitude (2^-40), a row with a single nonzero entry and an all-zero row. The experts
    have power-of-two row scales, so their dequantised weights are exact BF16 values and
    the BF16 block on those weights computes the same products: the FP8 block must agree
    with it to within two BF16 steps of each row's largest output, and both must match the
    oracle to the output tolerance's Frobenius bound row by row. (With such outliers the
    BF16 rounding of h and y, which both blocks share, exceeds the per-element bound on
    elements that cancel, so that bound is checked on the ordinary rows only.)"""
    import pins
    from oracle import oracle as O
    shape = W.TINY
    fp8, bf = pins._pow2_fp8_experts(shape, 3)
    q8 = tuple((q.cuda(), s.cuda()) for q, s in fp8)
    wg, wu, wd = (w.cuda() for w in bf)
    T = 40
    x = W.make_tokens(shape, T, 8, "cuda").float()
    x[0:8, 3] = 4096.0
    x[8:16, 100:110] = -3000.0
    x[16:24] *= 2.0 ** -40
    x[24] = 0.0
    x[24, 7] = 1.5
    x[25] = 0.0
    x = x.to(torch.bfloat16)
    wr, b = W.make_router(shape, 8, "cuda")
    o8 = moe.forward_fp8(x, wr, b, q8, shape).double().cpu().numpy()
    o16 = moe.forward(x, wr, b, wg, wu, wd, shape).double().cpu().numpy()
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    abi.beam_moe_device_status()
    experts = lambda e: (O.bf16_bits(bf[0][e]), O.bf16_bits(bf[1][e]), O.bf16_bits(bf[2][e]))  # noqa: E731
    ref, _, _ = O.forward(shape, O.bf16_bits(x), b.cpu().numpy(), experts, logits=logits)
    assert np.all(o8[25] == 0.0) and np.all(o16[25] == 0.0)
    for t in range(T):
        if t == 25:
            continue
        top = np.abs(o16[t]).max()
        assert np.abs(o8[t] - o16[t]).max() <= 2.0 ** -7 * top, t
        for o in (o8, o16):
            assert np.linalg.norm(o[t] - ref[t]) <= P.FROB * np.linalg.norm(ref[t]), t
    P.check_output(o8[16:], ref[16:], "wide-range activations, ordinary rows")


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
    cache = {}
    run_and_check(shape, x, wr, b, beam_fp8, tokens, f"{name} fp8 T={T}", cache)
    if T >= 1024:
        # the expert with the most rows is split evenly over N-tiles of at most 128 rows, all
        # but the last holding more than 64: one token every 64 of its rows and its last
        idx, _ = moe.route(x, wr, b, shape)
        idx = idx.cpu().numpy()
        load = np.bincount(idx.ravel(), minlength=shape.E)
        hottest = int(load.argmax())
        rows = np.nonzero((idx == hottest).any(axis=1))[0]
        pick = np.unique(np.concatenate([rows[::64], rows[-1:]]))
        run_and_check(shape, x, wr, b, beam_fp8, pick, f"{name} fp8 expert {hottest} ({load.max()} rows)", cache)
