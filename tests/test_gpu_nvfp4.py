"""NVFP4 expert weights: the CUDA block with E2M1 codes, E4M3 block scales and FP32 tensor
scales against the oracle on the same codes and scales (forward_nvfp4), element by
element, on Tiny (every token, ragged counts, both N-tile sizes of the NVFP4 kernel: 16 rows
while experts average at most 8 rows, else 32) and on Beam shapes (sampled tokens at full
size), plus a case that puts every E2M1 code and a wide range of block scales through the
block-scaled FP4 products."""
import numpy as np
import pytest
import torch

import parity as P
from oracle import oracle as O
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def host_experts(q4, cache=None):
    """Oracle callable e -> (gate, up, down), each (codes, block scales, tensor scale), over
    device NVFP4 experts, copying an expert to the host on first use."""
    cache = {} if cache is None else cache

    def get(e):
        if e not in cache:
            cache[e] = tuple((q[e].cpu().numpy(), bs[e].cpu().numpy(), float(t[e])) for q, bs, t in q4)
        return cache[e]
    return get


def run_and_check(shape, x, wr, b, q4, tokens, what, cache=None):
    out = moe.forward_nvfp4(x, wr, b, q4, shape)
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    idx, _ = moe.route(x, wr, b, shape)
    abi.beam_moe_device_status()
    out = out.float().cpu().numpy()
    tokens = np.asarray(tokens, np.int64)
    bh = b.cpu().numpy()
    _, _, dbg = O.route(shape, logits[tokens], bh, debug=True)
    flagged = P.near_tie_tokens(shape, dbg)
    experts = host_experts(q4, cache)
    ref, _ = O.forward_nvfp4(shape, O.bf16_bits(x), bh, experts, tokens, logits=logits)
    if len(flagged):
        ref2, _ = O.forward_nvfp4(shape, O.bf16_bits(x), bh, experts, tokens[flagged], logits=logits,
                                  idx_in=idx.cpu().numpy()[tokens[flagged]])
        ref[flagged] = ref2
    frob = P.check_output(out[tokens], ref, what)
    print(f"{what}: tokens checked {len(tokens)}, near-tie {len(flagged)}, rel frob {frob:.2e}")
    return out


@pytest.fixture(scope="module")
def tiny_fp4():
    return W.make_experts_nvfp4(W.TINY, seed=0, device="cuda")


@pytest.mark.parametrize("T", [1, 16, 33, 129, 300, 1500])
def test_tiny_nvfp4_parity(tiny_fp4, T):
    shape = W.TINY
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    run_and_check(shape, x, wr, b, tiny_fp4, np.arange(T), f"tiny nvfp4 T={T}")


def test_every_code_and_a_wide_range_of_block_scales():
    """Codes cycle through all 16 E2M1 values and block scales cover the E4M3 codes from the
    subnormal 2^-9 to 448 (h then spans about 1e-3 to 1.1e3 in magnitude). The block must
    match the oracle row by row to the output tolerance's Frobenius bound. (Block scales 2^18
    apart make some outputs cancel far below their terms, where the BF16 rounding of the
    output exceeds the per-element bound.) The same weights are exact in BF16 (tensor scales
    are powers of two), so the BF16 block on them is held to the same bound: a sanity check
    of the case itself."""
    import pins
    shape = W.TINY
    E, d, I = shape.E, shape.d, shape.I
    gen = torch.Generator().manual_seed(17)

    def part(rows, cols):
        q = torch.randint(0, 256, (E, rows, cols // 2), generator=gen, dtype=torch.int32).to(torch.uint8)
        bs = torch.randint(1, 127, (E, rows, cols // 16), generator=gen, dtype=torch.int32).to(torch.uint8)
        t = torch.full((E,), 2.0 ** -10, dtype=torch.float32)
        return q, bs, t

    parts = (part(I, d), part(I, d), part(d, I))
    deq = [torch.stack([pins.nvfp4_dequant_torch(q[e], bs[e], t[e]) for e in range(E)]) for q, bs, t in parts]
    wbf = [w.to(torch.bfloat16) for w in deq]
    for w, wb in zip(deq, wbf):
        assert torch.equal(wb.double(), w)
    q4 = tuple((q.cuda(), bs.cuda(), t.cuda()) for q, bs, t in parts)
    T = 40
    x = W.make_tokens(shape, T, 4, "cuda")
    wr, b = W.make_router(shape, 4, "cuda")
    o4 = moe.forward_nvfp4(x, wr, b, q4, shape).double().cpu().numpy()
    o16 = moe.forward(x, wr, b, *(w.cuda() for w in wbf), shape).double().cpu().numpy()
    logits = moe.router_logits(x, wr, shape).cpu().numpy()
    abi.beam_moe_device_status()
    experts = lambda e: (O.bf16_bits(wbf[0][e]), O.bf16_bits(wbf[1][e]), O.bf16_bits(wbf[2][e]))  # noqa: E731
    ref, _, _ = O.forward(shape, O.bf16_bits(x), b.cpu().numpy(), experts, logits=logits)
    for t in range(T):
        assert np.linalg.norm(o4[t] - ref[t]) <= P.FROB * np.linalg.norm(ref[t]), t
        assert np.linalg.norm(o16[t] - ref[t]) <= P.FROB * np.linalg.norm(ref[t]), t


def test_activation_blocks_beyond_the_first_piece_are_flagged():
    """A token block whose largest magnitude exceeds 6 * 448 cannot be carried by the first
    piece: the block clamps it and records status code 4; smaller blocks leave no status.
    (Tensor scales shrunk by 2^-10 keep h far inside the range.)"""
    shape = W.TINY
    q4 = tuple((q, bs, t * 2.0 ** -10) for q, bs, t in W.make_experts_nvfp4(shape, seed=3, device="cuda"))
    x = W.make_tokens(shape, 8, 5, "cuda")
    wr, b = W.make_router(shape, 5, "cuda")
    abi.beam_moe_device_status()
    x_ok = x.clone()
    x_ok[3, 17] = 2600.0
    moe.forward_nvfp4(x_ok, wr, b, q4, shape)
    abi.beam_moe_device_status()
    x_big = x.clone()
    x_big[3, 17] = 3000.0
    moe.forward_nvfp4(x_big, wr, b, q4, shape)
    with pytest.raises(abi.BeamMoeError) as err:
        abi.beam_moe_device_status()
    assert err.value.code == abi.BEAM_MOE_ERR_DEVICE and "2688" in str(err.value)


def test_nvfp4_deterministic(tiny_fp4):
    shape = W.TINY
    x = W.make_tokens(shape, 300, 7, "cuda")
    wr, b = W.make_router(shape, 7, "cuda")
    a = moe.forward_nvfp4(x, wr, b, tiny_fp4, shape)
    c = moe.forward_nvfp4(x, wr, b, tiny_fp4, shape)
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_nvfp4_close_to_bf16_block(tiny_fp4):
    """Same draws as the BF16 experts, quantised to NVFP4: the blocks differ by the
    quantisation error (about 10% relative per weight, averaging out over the sums)."""
    shape = W.TINY
    x = W.make_tokens(shape, 200, 1, "cuda")
    wr, b = W.make_router(shape, 1, "cuda")
    wg, wu, wd = W.make_experts(shape, 0, "cuda")
    ref = moe.forward(x, wr, b, wg, wu, wd, shape).double()
    got = moe.forward_nvfp4(x, wr, b, tiny_fp4, shape).double()
    rel = float((got - ref).norm() / ref.norm())
    assert rel < 0.2, rel


def test_nvfp4_rejects_shapes_off_the_block_grid():
    shape = W.MoEShape(d=384, I=256)
    x = torch.zeros((4, shape.d), dtype=torch.bfloat16, device="cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    q4 = tuple((torch.zeros((shape.E, r, c // 2), dtype=torch.uint8, device="cuda"),
                torch.zeros((shape.E, r, c // 16), dtype=torch.uint8, device="cuda"),
                torch.ones((shape.E,), dtype=torch.float32, device="cuda"))
               for r, c in ((shape.I, shape.d), (shape.I, shape.d), (shape.d, shape.I)))
    with pytest.raises(abi.BeamMoeError) as err:
        moe.forward_nvfp4(x, wr, b, q4, shape)
    assert err.value.code == abi.BEAM_MOE_ERR_ARG and "multiples of 256" in str(err.value)


@pytest.fixture(scope="module")
def beam_fp4():
    return W.make_experts_nvfp4(W.BEAM, seed=0, device="cuda")


@pytest.mark.parametrize("name,T,n_check", [("decode", 16, 16), ("prefill", 4096, 8)])
def test_beam_nvfp4_parity(beam_fp4, name, T, n_check):
    shape = W.BEAM
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    tokens = W.sample_tokens(T, n_check, seed=2).numpy()
    if T > n_check:
        tokens = np.unique(np.concatenate([tokens, [T - 1]]))
    cache = {}
    run_and_check(shape, x, wr, b, beam_fp4, tokens, f"{name} nvfp4 T={T}", cache)
    if T >= 64:
        # the expert with the most rows is split over several N-tiles of at most 32 rows: one
        # token every 16 of its rows hits each of them but the last, which its last row hits
        idx, _ = moe.route(x, wr, b, shape)
        idx = idx.cpu().numpy()
        load = np.bincount(idx.ravel(), minlength=shape.E)
        hottest = int(load.argmax())
        rows = np.nonzero((idx == hottest).any(axis=1))[0]
        pick = np.unique(np.concatenate([rows[::16], rows[-1:]]))
        run_and_check(shape, x, wr, b, beam_fp4, pick, f"{name} nvfp4 expert {hottest} ({load.max()} rows)", cache)
