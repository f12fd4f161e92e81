"""Checks that pin the CPU oracle to facts fixed outside itself.

Each check takes a loaded oracle build and raises AssertionError when the oracle breaks
the fact it pins. The same checks run against the real oracle (tests/test_oracle_pins.py)
and against copies of it with planted mistakes (tests/test_oracle_mutants.py), which must
each fail at least one check.

What pins what:
  * hand-worked routing cases (tests/golden/routing_handworked.json): group rule,
    masking of dropped groups, tie order, bias for selection only, weights;
  * brute force over all C(n_group, topk_group) group subsets and all top_k subsets of
    the candidates (small configs): the selection maximises the ranked sums;
  * reductions to library routines: torch.topk for group top-2 sums and for the plain
    top-k case; scipy's expit for the sigmoid; numpy FP64 matmul for the logits;
    torch float64 matmuls + torch.nn.functional.silu for the SwiGLU experts;
  * invariants: distinct experts inside kept groups, weights > 0 summing to the scale;
  * closed forms: all-zero input -> experts 0..7, weights scale/8, output 0; identical
    experts -> output = scale * expert(x).
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special
import torch

from sparse_moe_transformer_bias_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "routing_handworked.json")
E2M1_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e2m1_values.json")


def small_shape(**kw):
    base = dict(d=48, I=40, E=16, n_group=4, topk_group=2, top_k=3, scale=2.5)
    base.update(kw)
    return W.MoEShape(**base)


def random_routing_inputs(shape, T, seed=0, logit_std=1.0):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((T, shape.E)) * logit_std).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, shape.E).astype(np.float32)
    return logits, bias


def tiny_layer(seed=0, T=24, shape=W.TINY):
    x = W.make_tokens(shape, T, seed)
    wr, b = W.make_router(shape, seed)
    wg, wu, wd = W.make_experts(shape, seed)
    return x, wr, b, wg, wu, wd


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _torch_expert(x64, wg, wu, wd):
    """SwiGLU expert with torch float64 ops: down(silu(gate x) * up x)."""
    g = x64 @ wg.double().T
    u = x64 @ wu.double().T
    return (torch.nn.functional.silu(g) * u) @ wd.double().T


# ----------------------------------------------------------------------------------------

def check_golden_cases(orc):
    spec = json.load(open(GOLDEN))
    c = spec["config"]
    shape = W.MoEShape(d=8, I=8, E=c["E"], n_group=c["n_group"], topk_group=c["topk_group"], top_k=c["top_k"],
                       scale=c["scale"])
    for case in spec["cases"]:
        bias = np.full(shape.E, case["default_bias"], np.float32)
        for e, v in case["bias"].items():
            bias[int(e)] = v
        for tok in case["tokens"]:
            l = np.full((1, shape.E), tok["default_logit"], np.float32)
            for e, v in tok["logits"].items():
                l[0, int(e)] = v
            idx, w, dbg = orc.route(shape, l, bias, debug=True)
            assert list(dbg["groups"][0]) == tok["expect_groups"], (case["name"], dbg["groups"][0])
            assert list(idx[0]) == tok["expect_idx"], (case["name"], idx[0])
            np.testing.assert_allclose(w[0], tok["expect_w"], rtol=2e-6, err_msg=case["name"])


def check_invariants(orc, shape=W.BEAM, T=3000, seed=1):
    logits, bias = random_routing_inputs(shape, T, seed, logit_std=1.5)
    idx, w, dbg = orc.route(shape, logits, bias, debug=True)
    S = shape.E // shape.n_group
    for t in range(T):
        ids = idx[t]
        assert len(set(ids.tolist())) == shape.top_k, ("duplicate expert", t, ids)
        kept = set(dbg["groups"][t].tolist())
        assert len(kept) == shape.topk_group
        assert all((e // S) in kept for e in ids), ("expert outside kept groups", t)
        # every picked score >= every unpicked candidate score of the kept groups
        cand = [e for e in range(shape.E) if (e // S) in kept and e not in set(ids.tolist())]
        cmin = min(dbg["c"][t, ids])
        assert all(dbg["c"][t, e] <= cmin for e in cand), ("unpicked candidate beats a pick", t)
        # descending slot order
        cs = dbg["c"][t, ids]
        assert np.all(cs[:-1] >= cs[1:]), ("slot order", t)
    assert np.all(w > 0)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), shape.scale, rtol=2e-6)
    np.testing.assert_allclose(dbg["w64"].sum(1), shape.scale, rtol=1e-12)


def check_sigmoid_and_bias(orc, shape=W.BEAM, T=500, seed=2):
    logits, bias = random_routing_inputs(shape, T, seed, logit_std=3.0)
    _, _, dbg = orc.route(shape, logits, bias, debug=True)
    ref = scipy.special.expit(logits.astype(np.float64)).astype(np.float32)
    ulps = np.abs(dbg["s"].view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1 and (ulps > 0).mean() < 1e-3, ("sigmoid", ulps.max(), (ulps > 0).mean())
    # biased score: one FP32 add of the rounded sigmoid and the bias
    np.testing.assert_array_equal(dbg["c"], (dbg["s"] + bias[None, :]).astype(np.float32))


def check_group_scores_vs_topk(orc, shape=W.BEAM, T=500, seed=3):
    logits, bias = random_routing_inputs(shape, T, seed)
    _, _, dbg = orc.route(shape, logits, bias, debug=True)
    c = torch.from_numpy(dbg["c"]).view(T, shape.n_group, shape.E // shape.n_group)
    top2 = torch.topk(c, 2, dim=-1).values
    ref = (top2[..., 0] + top2[..., 1]).numpy()
    np.testing.assert_array_equal(dbg["gs"], ref)


def check_group_choice_brute_force(orc, shape=W.BEAM, T=400, seed=4):
    logits, bias = random_routing_inputs(shape, T, seed)
    _, _, dbg = orc.route(shape, logits, bias, debug=True)
    subsets = list(itertools.combinations(range(shape.n_group), shape.topk_group))
    for t in range(T):
        gs = dbg["gs"][t].astype(np.float64)
        best = max(subsets, key=lambda sub: (sum(gs[g] for g in sub), [-g for g in sub]))
        assert set(best) == set(dbg["groups"][t].tolist()), (t, best, dbg["groups"][t])


def check_selection_brute_force_small(orc, T=300, seed=5):
    """Small config: enumerate all group subsets, then all top_k subsets of the kept
    candidates; the oracle's picks must be the best subset by (group score sum, then
    biased score sum)."""
    shape = small_shape()
    logits, bias = random_routing_inputs(shape, T, seed)
    idx, _, dbg = orc.route(shape, logits, bias, debug=True)
    S = shape.E // shape.n_group
    s64 = scipy.special.expit(logits.astype(np.float64)).astype(np.float32)
    for t in range(T):
        c = (s64[t] + bias).astype(np.float32).astype(np.float64)
        gs = [sum(sorted(c[g * S:(g + 1) * S], reverse=True)[:2]) for g in range(shape.n_group)]
        kept = max(itertools.combinations(range(shape.n_group), shape.topk_group), key=lambda sub: sum(gs[g] for g in sub))
        cand = [e for e in range(shape.E) if e // S in kept]
        picks = max(itertools.combinations(cand, shape.top_k), key=lambda sub: sum(c[e] for e in sub))
        assert set(picks) == set(idx[t].tolist()), (t, picks, idx[t])


def check_plain_topk_reduction(orc, T=300, seed=6):
    """All groups kept and zero bias: routing is torch.topk of the logits (sigmoid is
    monotone), also with a single group."""
    for shape in (W.MoEShape(d=8, I=8, topk_group=8), W.MoEShape(d=8, I=8, n_group=1, topk_group=1)):
        logits, _ = random_routing_inputs(shape, T, seed)
        bias = np.zeros(shape.E, np.float32)
        idx, _ = orc.route(shape, logits, bias)
        ref = torch.topk(torch.from_numpy(logits), shape.top_k, dim=1).indices.numpy()
        np.testing.assert_array_equal(idx, ref)


def check_logits_vs_matmul(orc, seed=7):
    shape = W.TINY
    x = W.make_tokens(shape, 64, seed)
    wr, _ = W.make_router(shape, seed)
    l = orc.router_logits(shape, _bits(x), wr.numpy())
    ref = (x.double().numpy() @ wr.double().numpy().T).astype(np.float32)
    ulps = np.abs(l.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1, ulps.max()


def check_expert_vs_torch(orc, seed=8):
    shape = W.TINY
    x, _, _, wg, wu, wd = tiny_layer(seed, T=4)
    for t, e in ((0, 3), (1, 200), (3, 77)):
        y = orc.expert(shape, x[t].double().numpy(), _bits(wg[e]), _bits(wu[e]), _bits(wd[e]))
        ref = _torch_expert(x[t:t + 1].double(), wg[e], wu[e], wd[e])[0].numpy()
        np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def check_forward_combination(orc, seed=9):
    """Forward = sum_k w_k * expert_{e_k}(x), with the weights re-derived from scipy's
    sigmoid of the logits and the experts from torch float64 ops."""
    shape = W.TINY
    x, wr, b, wg, wu, wd = tiny_layer(seed, T=12)
    out, idx, w = orc.forward(shape, _bits(x), b.numpy(), lambda e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e])),
                              router_w=wr.numpy())
    logits = orc.router_logits(shape, _bits(x), wr.numpy())
    s = scipy.special.expit(logits.astype(np.float64)).astype(np.float32).astype(np.float64)
    for t in range(x.shape[0]):
        ws = s[t, idx[t]]
        ws = shape.scale * ws / ws.sum()
        np.testing.assert_allclose(w[t], ws, rtol=2e-6)
        ref = sum(ws[k] * _torch_expert(x[t:t + 1].double(), wg[idx[t, k]], wu[idx[t, k]], wd[idx[t, k]])[0]
                  for k in range(shape.top_k)).numpy()
        np.testing.assert_allclose(out[t], ref, rtol=1e-9, atol=1e-12)


def check_zero_input(orc, seed=10):
    shape = W.TINY
    _, wr, _, wg, wu, wd = tiny_layer(seed, T=1)
    x = torch.zeros((3, shape.d), dtype=torch.bfloat16)
    b = np.full(shape.E, 0.037, np.float32)
    out, idx, w = orc.forward(shape, _bits(x), b, lambda e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e])),
                              router_w=wr.numpy())
    assert (idx == np.arange(8)[None, :]).all(), idx
    assert (w == np.float32(shape.scale / 8)).all(), w
    assert (out == 0).all()


def check_identical_experts(orc, seed=11):
    shape = W.TINY
    x, wr, b, wg, wu, wd = tiny_layer(seed, T=6)
    one = (_bits(wg[5]), _bits(wu[5]), _bits(wd[5]))
    out, _, _ = orc.forward(shape, _bits(x), b.numpy(), lambda e: one, router_w=wr.numpy())
    ref = shape.scale * _torch_expert(x.double(), wg[5], wu[5], wd[5]).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def check_given_selection(orc, seed=12):
    """With the selection handed in, the oracle uses exactly those experts and re-derives
    their weights from its own sigmoid scores."""
    shape = W.TINY
    x, wr, b, wg, wu, wd = tiny_layer(seed, T=3)
    experts = lambda e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e]))
    pick = np.array([[7, 6, 5, 4, 3, 2, 1, 0], [255, 0, 128, 64, 32, 16, 8, 4], [10, 11, 12, 13, 14, 15, 16, 17]],
                    np.int32)
    out, idx, w = orc.forward(shape, _bits(x), b.numpy(), experts, router_w=wr.numpy(), idx_in=pick)
    assert (idx == pick).all()
    logits = orc.router_logits(shape, _bits(x), wr.numpy())
    s = scipy.special.expit(logits.astype(np.float64)).astype(np.float32).astype(np.float64)
    for t in range(3):
        ws = shape.scale * s[t, pick[t]] / s[t, pick[t]].sum()
        np.testing.assert_allclose(w[t], ws, rtol=2e-6)


# ---------------------------------------------------------------- sandwich norm and residual

def pin_rmsnorm_library(O):
    """RMSNorm equals torch.nn.functional.rms_norm in float64 (an independent library
    routine), for several widths, scales and eps."""
    rng = np.random.default_rng(11)
    for d, scale, eps in ((8, 1.0, 1e-6), (512, 3.0, 1e-5), (5120, 0.02, 1e-6), (96, 1e-3, 1e-2)):
        v = rng.standard_normal(d) * scale
        gamma = torch.randn(d, dtype=torch.float32).to(torch.bfloat16)
        got = O.rmsnorm(v, _bits(gamma), eps)
        want = torch.nn.functional.rms_norm(torch.from_numpy(v), (d,), weight=gamma.double(), eps=eps).numpy()
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


def pin_rmsnorm_closed_forms(O):
    """Constant row c: gamma * c / sqrt(c^2 + eps). Scale invariance: rmsnorm(s v) =
    rmsnorm(v) when eps = 0. Unit gain on a row of RMS 1 with eps = 0: the row itself."""
    d = 64
    gamma = torch.full((d,), 1.5, dtype=torch.bfloat16)
    for c in (-2.0, 0.25, 7.0):
        got = O.rmsnorm(np.full(d, c), _bits(gamma), 1e-3)
        np.testing.assert_allclose(got, 1.5 * c / np.sqrt(c * c + 1e-3), rtol=1e-14)
    rng = np.random.default_rng(12)
    v = rng.standard_normal(d)
    g1 = torch.ones(d, dtype=torch.bfloat16)
    np.testing.assert_allclose(O.rmsnorm(37.0 * v, _bits(g1), 0.0), O.rmsnorm(v, _bits(g1), 0.0), rtol=1e-13)
    u = v / np.sqrt(np.mean(v * v))
    np.testing.assert_allclose(O.rmsnorm(u, _bits(g1), 0.0), u, rtol=1e-13)


def pin_residual_is_scaled_sum(O):
    """Depth-scaled residual: starting from the embedding (contribution 1) and adding
    contributions 2..K one step at a time gives the sum of all K divided by sqrt(K), the
    statement of the transformers doc; the stream keeps unit RMS when the contributions
    are orthonormal."""
    rng = np.random.default_rng(13)
    d, K = 32, 9
    parts = rng.standard_normal((K, d))
    stream = parts[0].copy()
    for k in range(2, K + 1):
        stream = O.residual(stream, parts[k - 1], k)
    np.testing.assert_allclose(stream, parts.sum(axis=0) / np.sqrt(K), rtol=1e-12, atol=1e-13)
    q, _ = np.linalg.qr(rng.standard_normal((d, K)))
    stream = q[:, 0] * np.sqrt(d)
    for k in range(2, K + 1):
        stream = O.residual(stream, q[:, k - 1] * np.sqrt(d), k)
        np.testing.assert_allclose(np.sqrt(np.mean(stream * stream)), 1.0, rtol=1e-12)


def pin_round_bf16_vs_torch(O):
    """The oracle's BF16 rounding equals torch's FP32 -> BF16 conversion (round to nearest,
    ties to even) on values that are exact in FP32, including exact ties."""
    rng = np.random.default_rng(14)
    v32 = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    ties = (np.float32(1.0) + np.arange(1, 200, dtype=np.float32) * np.float32(2.0 ** -8)).astype(np.float32)
    v32 = np.concatenate([v32, ties, -ties, np.float32([0.0, 1.0, -2.5, 65504.0])])
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.round_bf16(v32.astype(np.float64)), want)


def pin_sublayer_composition(O, seed=15):
    """Whole sublayer with identical experts (routing drops out: the MoE output is
    2.5 * expert(x)), against torch float64 in the pages' order: pre-RMSNorm, BF16 input,
    SwiGLU expert, x2.5, post-RMSNorm, depth-scaled residual with k = 7."""
    shape = W.TINY
    T, k, eps = 6, 7, 1e-6
    g = torch.Generator().manual_seed(seed)
    stream = torch.randn((T, shape.d), generator=g).mul_(3.0).to(torch.bfloat16)
    pre = (1.0 + 0.1 * torch.randn(shape.d, generator=g)).to(torch.bfloat16)
    post = (1.0 + 0.1 * torch.randn(shape.d, generator=g)).to(torch.bfloat16)
    wr, b = W.make_router(shape, seed)
    wg1, wu1, wd1 = (w[3] for w in W.make_experts(shape, seed))
    experts = lambda e: (_bits(wg1), _bits(wu1), _bits(wd1))  # noqa: E731
    out, _ = O.sublayer(shape, _bits(stream), _bits(pre), _bits(post), eps, k, b.numpy(), experts,
                        np.arange(T), router_w=wr.numpy())
    s64 = stream.double()
    x = torch.nn.functional.rms_norm(s64, (shape.d,), weight=pre.double(), eps=eps).float().to(torch.bfloat16)
    m = 2.5 * _torch_expert(x.double(), wg1, wu1, wd1)
    y = torch.nn.functional.rms_norm(m, (shape.d,), weight=post.double(), eps=eps)
    want = math.sqrt((k - 1) / k) * s64 + y / math.sqrt(k)
    np.testing.assert_allclose(out, want.numpy(), rtol=1e-9, atol=1e-9)


def pin_forward_grouped_vs_per_token(O, seed=17):
    """The grouped evaluation (numpy FP64 products per expert) equals the per-token C
    forward, with the oracle's own routing and with a given selection."""
    shape = W.TINY
    x = W.make_tokens(shape, 48, seed, "cpu")
    wr, b = W.make_router(shape, seed, "cpu")
    wg, wu, wd = W.make_experts(shape, seed, "cpu")
    xb = _bits(x)
    host = {e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e])) for e in range(shape.E)}
    experts = host.get
    tokens = np.array([0, 3, 4, 9, 17, 30, 47])
    logits = O.router_logits(shape, xb, wr.numpy())
    ref, idx_r, _ = O.forward(shape, xb, b.numpy(), experts, tokens=tokens, logits=logits)
    got, idx_g = O.forward_grouped(shape, xb, b.numpy(), experts, tokens, logits=logits)
    assert np.array_equal(idx_r, idx_g)
    assert np.abs(got - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1.0)
    sel = np.roll(idx_r, 1, axis=1)  # a different slot order of the same experts
    ref2, _, _ = O.forward(shape, xb, b.numpy(), experts, tokens=tokens, logits=logits, idx_in=sel)
    got2, _ = O.forward_grouped(shape, xb, b.numpy(), experts, tokens, logits=logits, idx_in=sel)
    assert np.abs(got2 - ref2).max() <= 1e-12 * max(np.abs(ref2).max(), 1.0)
    # the sublayer with its MoE block evaluated the grouped way
    g = torch.Generator().manual_seed(seed)
    stream = torch.randn((48, shape.d), generator=g).mul_(3.0).to(torch.bfloat16)
    gain = (1.0 + 0.1 * torch.randn(shape.d, generator=g)).to(torch.bfloat16)
    args = (shape, _bits(stream), _bits(gain), _bits(gain), 1e-6, 5, b.numpy(), experts, tokens)
    ref3, _ = O.sublayer(*args, router_w=wr.numpy())
    got3, _ = O.sublayer(*args, router_w=wr.numpy(), grouped=True)
    assert np.abs(got3 - ref3).max() <= 1e-12 * max(np.abs(ref3).max(), 1.0)


def pin_e4m3_decoder_vs_torch(O):
    """Every FP8 E4M3 code decodes to torch's float8_e4m3fn value (NaN codes to NaN)."""
    q = np.arange(256, dtype=np.uint8)
    got = O.e4m3_decode(q)
    want = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_array_equal(got[~np.isnan(got)], want[~np.isnan(want)])


def pin_fp8_expert_vs_torch(O, seed=16):
    """The FP8 expert equals the BF16-free SwiGLU of torch float64 on the dequantised
    weights (per-row scale times the E4M3 value), for the quantised Tiny experts."""
    shape = W.TINY
    (gq, gs), (uq, us), (dq, ds) = W.make_experts_fp8(shape, seed)
    e = 5
    deq = lambda q, sc: torch.from_numpy(O.e4m3_decode(q[e].numpy())) * sc[e].double().unsqueeze(1)  # noqa: E731
    wg64, wu64, wd64 = deq(gq, gs), deq(uq, us), deq(dq, ds)
    x = torch.randn(shape.d, generator=torch.Generator().manual_seed(seed), dtype=torch.float64)
    got = O.expert_fp8(shape, x.numpy(), gq[e].numpy(), gs[e].numpy(), uq[e].numpy(), us[e].numpy(), dq[e].numpy(),
                       ds[e].numpy())
    want = (torch.nn.functional.silu(wg64 @ x) * (wu64 @ x)) @ wd64.T
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)
    # and the quantisation is close to the BF16 expert it came from (a sanity bound)
    wg, wu, wd = (w[e].double() for w in W.make_experts(shape, seed))
    ref = (torch.nn.functional.silu(wg @ x) * (wu @ x)) @ wd.T
    assert float((want - ref).norm() / ref.norm()) < 0.08



def _pow2_fp8_experts(shape, seed):
    """FP8 experts whose dequantised weights are exact BF16 values: per-row scales that are
    powers of two (2^ceil(log2(absmax / 448))), codes rounded to E4M3 by torch. An E4M3
    value has at most 4 significant bits, so scale * value is a BF16 number. Returns the
    codes and scales as ((gq, gs), (uq, us), (dq, ds)) and the equal BF16 experts."""
    g = torch.Generator().manual_seed(seed)
    fp8, bf = [], []
    for rows, cols in ((shape.I, shape.d), (shape.I, shape.d), (shape.d, shape.I)):
        w = torch.randn((shape.E, rows, cols), generator=g, dtype=torch.float64) / math.sqrt(cols)
        amax = w.abs().amax(dim=-1).clamp_min(1e-30)
        sc = torch.exp2(torch.ceil(torch.log2(amax / W.FP8_MAX))).float()
        q = (w / sc.double().unsqueeze(-1)).float().to(torch.float8_e4m3fn)
        deq = q.to(torch.float64) * sc.double().unsqueeze(-1)
        wb = deq.to(torch.bfloat16)
        assert torch.equal(wb.double(), deq), "a power-of-two-scaled E4M3 weight must be a BF16 value"
        fp8.append((q.view(torch.uint8), sc))
        bf.append(wb)
    return tuple(fp8), tuple(bf)


def pin_forward_fp8_equals_bf16_block(orc, seed=18):
    """The FP8 block's composition (routing, weights, slot sum) against the BF16 block: on
    FP8 experts whose dequantised weights are exactly BF16 values, forward_fp8 must equal
    forward on those BF16 weights, both with the oracle's own routing and with a selection
    handed in (weights re-derived from the unbiased sigmoid scores)."""
    shape = W.MoEShape(d=64, I=48)  # Beam's routing (256 experts, 8 groups, top 4, top 8), narrow experts
    T = 6
    x = W.make_tokens(shape, T, seed)
    wr, b = W.make_router(shape, seed)
    ((gq, gs), (uq, us), (dq, ds)), (wg, wu, wd) = _pow2_fp8_experts(shape, seed)
    xb = _bits(x)
    experts_q = lambda e: (gq[e].numpy(), gs[e].numpy(), uq[e].numpy(), us[e].numpy(), dq[e].numpy(),  # noqa: E731
                           ds[e].numpy())
    experts_b = lambda e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e]))  # noqa: E731
    tokens = np.arange(T)
    logits = orc.router_logits(shape, xb, wr.numpy())
    ref, idx_r, _ = orc.forward(shape, xb, b.numpy(), experts_b, tokens=tokens, logits=logits)
    got, idx_g = orc.forward_fp8(shape, xb, b.numpy(), experts_q, tokens, logits=logits)
    np.testing.assert_array_equal(idx_g, idx_r)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # a selection from outside, in another slot order, with experts the router did not pick
    sel = np.roll(idx_r, 3, axis=1).copy()
    sel[:, 0] = (sel[:, 0] + 101) % shape.E
    for t in range(T):
        assert len(set(sel[t].tolist())) == shape.top_k
    ref2, _, _ = orc.forward(shape, xb, b.numpy(), experts_b, tokens=tokens, logits=logits, idx_in=sel)
    got2, idx2 = orc.forward_fp8(shape, xb, b.numpy(), experts_q, tokens, logits=logits, idx_in=sel)
    np.testing.assert_array_equal(idx2, sel)
    np.testing.assert_allclose(got2, ref2, rtol=1e-12, atol=1e-12 * np.abs(ref2).max())


def pin_forward_fp8_identical_experts(orc, seed=19):
    """Closed form for the FP8 block: when every expert is the same FP8 expert, the routed
    weights sum to the scale and the output is scale * expert_fp8(x), whatever the routing
    (router weights drawn from the Tiny recipe, FP8 experts from the quantisation recipe)."""
    shape = W.TINY
    T = 5
    x = W.make_tokens(shape, T, seed)
    wr, b = W.make_router(shape, seed)
    (gq, gs), (uq, us), (dq, ds) = W.make_experts_fp8(shape, seed)
    e0 = 9
    one = (gq[e0].numpy(), gs[e0].numpy(), uq[e0].numpy(), us[e0].numpy(), dq[e0].numpy(), ds[e0].numpy())
    out, _ = orc.forward_fp8(shape, _bits(x), b.numpy(), lambda e: one, np.arange(T), router_w=wr.numpy())
    # the single expert from torch float64 on the dequantised weights
    deq = lambda q, sc: torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64) \
        * torch.from_numpy(sc).double().unsqueeze(1)  # noqa: E731
    wg64, wu64, wd64 = deq(one[0], one[1]), deq(one[2], one[3]), deq(one[4], one[5])
    x64 = x.double()
    want = shape.scale * ((torch.nn.functional.silu(x64 @ wg64.T) * (x64 @ wu64.T)) @ wd64.T)
    np.testing.assert_allclose(out, want.numpy(), rtol=1e-10, atol=1e-12)


def _e2m1_table():
    return torch.tensor(json.load(open(E2M1_GOLDEN))["values"], dtype=torch.float64)


def nvfp4_dequant_torch(q, bs, t):
    """NVFP4 weights [rows, cols] in float64 from codes [rows, cols/2] (element 2k in the low
    half of byte k), E4M3 block scales [rows, cols/16] and a tensor scale, with the golden
    E2M1 table and torch's float8_e4m3fn (no oracle code)."""
    q = torch.as_tensor(q)
    rows, half = q.shape
    codes = torch.stack([q & 15, q >> 4], dim=-1).reshape(rows, 2 * half).long()
    vals = _e2m1_table()[codes].reshape(rows, -1, 16)
    scales = torch.as_tensor(bs).view(torch.float8_e4m3fn).to(torch.float64).unsqueeze(-1)
    return (vals * scales).reshape(rows, 2 * half) * float(t)


def pin_e2m1_decoder_table(O):
    """Every E2M1 code decodes to the value the format's table gives (signed zero included)."""
    spec = json.load(open(E2M1_GOLDEN))
    got = O.e2m1_decode(np.asarray(spec["codes"], np.uint8))
    want = np.asarray(spec["values"], np.float64)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(want))


def pin_nvfp4_expert_vs_torch(O, seed=20):
    """The NVFP4 expert equals the SwiGLU of torch float64 on the weights dequantised here
    (golden E2M1 table, torch E4M3 block scales, tensor scale), for a quantised Tiny expert;
    and the quantisation stays near the BF16 expert it came from (a sanity bound)."""
    shape = W.TINY
    mats = W.make_experts_nvfp4(shape, seed)
    e = 11
    parts = [(m[0][e].numpy(), m[1][e].numpy(), float(m[2][e])) for m in mats]
    wg64, wu64, wd64 = (nvfp4_dequant_torch(*p) for p in parts)
    x = torch.randn(shape.d, generator=torch.Generator().manual_seed(seed), dtype=torch.float64)
    got = O.expert_nvfp4(shape, x.numpy(), *parts)
    want = (torch.nn.functional.silu(wg64 @ x) * (wu64 @ x)) @ wd64.T
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)
    wg, wu, wd = (w[e].double() for w in W.make_experts(shape, seed))
    ref = (torch.nn.functional.silu(wg @ x) * (wu @ x)) @ wd.T
    assert float((want - ref).norm() / ref.norm()) < 0.25


def _exact_nvfp4_experts(shape, seed):
    """NVFP4 experts whose dequantised weights are exact BF16 values: random codes over all
    16 E2M1 values, block scales among the E4M3 codes with exponent field 5..9 (2^-2 .. 2^2
    times 1..1.875), tensor scales powers of two. A product of an E2M1 value (2 significant
    bits), an E4M3 value (4) and a power of two has at most 6, so it is a BF16 number.
    Returns the NVFP4 parts per matrix and the equal BF16 experts."""
    g = torch.Generator().manual_seed(seed)
    parts, bf = [], []
    for rows, cols in ((shape.I, shape.d), (shape.I, shape.d), (shape.d, shape.I)):
        q = torch.randint(0, 256, (shape.E, rows, cols // 2), generator=g, dtype=torch.int32).to(torch.uint8)
        bs = ((torch.randint(5, 10, (shape.E, rows, cols // 16), generator=g) << 3) |
              torch.randint(0, 8, (shape.E, rows, cols // 16), generator=g)).to(torch.uint8)
        t = torch.exp2(torch.randint(-5, -2, (shape.E,), generator=g).float()) / math.sqrt(cols)
        t = torch.exp2(torch.round(torch.log2(t)))
        deq = torch.stack([nvfp4_dequant_torch(q[e], bs[e], t[e]) for e in range(shape.E)])
        wb = deq.to(torch.bfloat16)
        assert torch.equal(wb.double(), deq), "such an NVFP4 weight must be a BF16 value"
        parts.append((q, bs, t))
        bf.append(wb)
    return tuple(parts), tuple(bf)


def pin_forward_nvfp4_equals_bf16_block(orc, seed=21):
    """The NVFP4 block's composition against the BF16 block: on NVFP4 experts whose
    dequantised weights are exact BF16 values, forward_nvfp4 must equal forward on those
    BF16 weights, with the oracle's own routing and with a selection handed in."""
    shape = W.MoEShape(d=64, I=48)
    T = 5
    x = W.make_tokens(shape, T, seed)
    wr, b = W.make_router(shape, seed)
    parts, (wg, wu, wd) = _exact_nvfp4_experts(shape, seed)
    xb = _bits(x)
    experts_q = lambda e: tuple((p[0][e].numpy(), p[1][e].numpy(), float(p[2][e])) for p in parts)  # noqa: E731
    experts_b = lambda e: (_bits(wg[e]), _bits(wu[e]), _bits(wd[e]))  # noqa: E731
    tokens = np.arange(T)
    logits = orc.router_logits(shape, xb, wr.numpy())
    ref, idx_r, _ = orc.forward(shape, xb, b.numpy(), experts_b, tokens=tokens, logits=logits)
    got, idx_g = orc.forward_nvfp4(shape, xb, b.numpy(), experts_q, tokens, logits=logits)
    np.testing.assert_array_equal(idx_g, idx_r)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    sel = np.roll(idx_r, 2, axis=1).copy()
    sel[:, 1] = (sel[:, 1] + 77) % shape.E
    for t in range(T):
        assert len(set(sel[t].tolist())) == shape.top_k
    ref2, _, _ = orc.forward(shape, xb, b.numpy(), experts_b, tokens=tokens, logits=logits, idx_in=sel)
    got2, idx2 = orc.forward_nvfp4(shape, xb, b.numpy(), experts_q, tokens, logits=logits, idx_in=sel)
    np.testing.assert_array_equal(idx2, sel)
    np.testing.assert_allclose(got2, ref2, rtol=1e-12, atol=1e-12 * np.abs(ref2).max())


ALL_CHECKS = [
    check_golden_cases, check_invariants, check_sigmoid_and_bias, check_group_scores_vs_topk,
    check_group_choice_brute_force, check_selection_brute_force_small, check_plain_topk_reduction,
    check_logits_vs_matmul, check_expert_vs_torch, check_forward_combination, check_zero_input,
    check_identical_experts, check_given_selection,
    pin_rmsnorm_library, pin_rmsnorm_closed_forms, pin_residual_is_scaled_sum, pin_round_bf16_vs_torch,
    pin_sublayer_composition, pin_e4m3_decoder_vs_torch, pin_fp8_expert_vs_torch, pin_forward_grouped_vs_per_token,
    pin_forward_fp8_equals_bf16_block, pin_forward_fp8_identical_experts,
    pin_e2m1_decoder_table, pin_nvfp4_expert_vs_torch, pin_forward_nvfp4_equals_bf16_block,
]
