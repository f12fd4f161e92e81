"""Helpers for comparing the CUDA library with the CPU oracle on the same seeded inputs.

Acceptance (Beam MoE block):
  * router logits: |gpu - oracle| <= 1e-5 * sum_j |x_j w_j| + 1e-6 (FP32 accumulation
    against an FP64 sum rounded once);
  * routing: given the GPU's own FP32 logits, expert indices equal the oracle's bit for
    bit, except tokens whose ranked biased scores (top_k+1 candidates) or group scores
    (topk_group+1 groups) have a neighbouring gap below 1e-6: those are reported
    separately and accepted when the GPU's picks are tie-consistent with the oracle's
    scores (same picked scores within 1e-6, descending order within 1e-6);
  * weights: |gpu - oracle| <= 1e-6 * |oracle| + 1e-7;
  * output: |gpu - oracle| <= 1e-2 + 2e-2 |oracle| per element and relative Frobenius
    error <= 5e-3. Near-tie tokens are compared against the oracle rerun on the GPU's
    selection.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from oracle import oracle as O

TIE = 1e-6
ATOL, RTOL, FROB = 1e-2, 2e-2, 5e-3


@dataclasses.dataclass
class Layer:
    shape: object
    x: torch.Tensor
    wr: torch.Tensor
    b: torch.Tensor
    wg: torch.Tensor = None
    wu: torch.Tensor = None
    wd: torch.Tensor = None
    host_cache: dict = dataclasses.field(default_factory=dict)

    def experts(self, needed):
        """Oracle `experts` callable holding host copies of the needed experts only."""
        for e in needed:
            if e not in self.host_cache:
                self.host_cache[e] = (O.bf16_bits(self.wg[e]), O.bf16_bits(self.wu[e]), O.bf16_bits(self.wd[e]))
        cache = self.host_cache
        return lambda e: cache.get(e)


def near_tie_tokens(shape, dbg):
    """Tokens whose selection may legitimately differ by FP32 rounding of the sigmoid."""
    T = dbg["c"].shape[0]
    S = shape.E // shape.n_group
    gs = -np.sort(-dbg["gs"].astype(np.float64), axis=1)
    ng = min(shape.topk_group + 1, shape.n_group)
    g_gap = np.min(gs[:, :ng - 1] - gs[:, 1:ng], axis=1) if ng > 1 else np.full(T, np.inf)
    kept = np.zeros((T, shape.n_group), bool)
    np.put_along_axis(kept, dbg["groups"].astype(np.int64), True, axis=1)
    c = np.where(np.repeat(kept, S, axis=1), dbg["c"].astype(np.float64), -np.inf)
    cs = -np.sort(-c, axis=1)
    nk = min(shape.top_k + 1, int(kept[0].sum()) * S)
    cs = cs[:, :nk]
    finite = np.isfinite(cs[:, 1:])
    e_gap = np.where(finite, cs[:, :-1] - cs[:, 1:], np.inf).min(axis=1)
    return np.nonzero((g_gap < TIE) | (e_gap < TIE))[0]


def check_routing(shape, gpu_logits, bias, gpu_idx, gpu_w):
    """Returns (flagged token ids, oracle debug dict). Raises on any mismatch."""
    idx_o, w_o, dbg = O.route(shape, gpu_logits, bias, debug=True)
    flagged = near_tie_tokens(shape, dbg)
    ok = np.ones(gpu_idx.shape[0], bool)
    ok[flagged] = False
    np.testing.assert_array_equal(gpu_idx[ok], idx_o[ok], err_msg="expert indices differ on non-tie tokens")
    np.testing.assert_allclose(gpu_w[ok], w_o[ok], rtol=1e-6, atol=1e-7, err_msg="routing weights")
    S = shape.E // shape.n_group
    for t in flagged:
        cg = dbg["c"][t, gpu_idx[t]].astype(np.float64)
        co = dbg["c"][t, idx_o[t]].astype(np.float64)
        assert len(set(gpu_idx[t].tolist())) == shape.top_k
        assert np.all(np.abs(np.sort(cg) - np.sort(co)) <= TIE), (t, gpu_idx[t], idx_o[t])
        assert np.all(cg[:-1] - cg[1:] >= -TIE), (t, "slot order")
        # the picks lie in at most topk_group groups, each of which could be kept: its group
        # score is within TIE of the oracle's topk_group-th best
        groups = sorted(set((gpu_idx[t] // S).tolist()))
        assert len(groups) <= shape.topk_group, (t, groups)
        gs = dbg["gs"][t].astype(np.float64)
        cut = np.sort(gs)[::-1][shape.topk_group - 1]
        assert all(gs[g] >= cut - TIE for g in groups), (t, groups, gs)
        # and every pick beats every candidate of those groups that was left out (to TIE)
        cand = [e for g in groups for e in range(g * S, (g + 1) * S) if e not in set(gpu_idx[t].tolist())]
        if cand:
            assert dbg["c"][t, cand].astype(np.float64).max() <= cg.min() + TIE, (t, "a better candidate was left out")
    return flagged, dbg


def check_logits(shape, x, wr, gpu_logits):
    xb = O.bf16_bits(x)
    ref = O.router_logits(shape, xb, wr.cpu().numpy())
    mag = np.abs(x.float().cpu().numpy()) @ np.abs(wr.cpu().numpy()).T
    err = np.abs(gpu_logits.astype(np.float64) - ref)
    bound = 1e-5 * mag + 1e-6
    assert np.all(err <= bound), f"logit error {err.max()} above bound"
    return float((err / (mag + 1e-30)).max())


def check_output(gpu_out, ref_out, what=""):
    g = gpu_out.astype(np.float64)
    r = ref_out.astype(np.float64)
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max()}"
    frob = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert frob <= FROB, f"{what}: relative Frobenius error {frob}"
    return frob


def oracle_forward_for(layer: Layer, tokens, gpu_logits_full, gpu_idx_full, grouped=False):
    """Oracle output for `tokens` given the GPU's logits; near-tie tokens are rerun on the
    GPU's selection. grouped: evaluate with the oracle's grouped form (numpy FP64 products
    per expert, for large token samples). Returns (out [n, d] FP64, flagged tokens among
    `tokens`)."""
    shape = layer.shape
    tokens = np.asarray(tokens, np.int64)
    lg = gpu_logits_full[tokens]
    b = layer.b.cpu().numpy()
    idx_r, _, dbg = O.route(shape, lg, b, debug=True)
    flagged_local = near_tie_tokens(shape, dbg)
    idx_in = np.asarray(gpu_idx_full[tokens], np.int32).copy()
    needed = set(np.unique(idx_in).tolist()) | set(np.unique(idx_r).tolist())
    xb = O.bf16_bits(layer.x)
    experts = layer.experts(needed)
    if grouped:
        out, _ = O.forward_grouped(shape, xb, b, experts, tokens, logits=gpu_logits_full)
    else:
        out, _, _ = O.forward(shape, xb, b, experts, tokens=tokens, logits=gpu_logits_full)
    if len(flagged_local):
        if grouped:
            out2, _ = O.forward_grouped(shape, xb, b, experts, tokens[flagged_local], logits=gpu_logits_full,
                                        idx_in=idx_in[flagged_local])
        else:
            out2, _, _ = O.forward(shape, xb, b, experts, tokens=tokens[flagged_local], logits=gpu_logits_full,
                                   idx_in=idx_in[flagged_local])
        out[flagged_local] = out2
    return out, tokens[flagged_local]


def oracle_forward_fp8_for(shape, x, bias, experts_q, tokens, gpu_logits_full, gpu_idx_full):
    """oracle_forward_for with FP8 experts (experts_q: e -> (wg_q, gs, wu_q, us, wd_q, ds) as
    numpy arrays): the oracle's routing from the GPU's logits, near-tie tokens rerun on the
    GPU's selection. Returns (out [n, d] FP64, flagged tokens among `tokens`)."""
    tokens = np.asarray(tokens, np.int64)
    b = bias.cpu().numpy()
    _, _, dbg = O.route(shape, gpu_logits_full[tokens], b, debug=True)
    flagged_local = near_tie_tokens(shape, dbg)
    xb = O.bf16_bits(x)
    out, _ = O.forward_fp8(shape, xb, b, experts_q, tokens, logits=gpu_logits_full)
    if len(flagged_local):
        idx_in = np.asarray(gpu_idx_full[tokens], np.int32)[flagged_local]
        out2, _ = O.forward_fp8(shape, xb, b, experts_q, tokens[flagged_local], logits=gpu_logits_full,
                                idx_in=idx_in)
        out[flagged_local] = out2
    return out, tokens[flagged_local]
