"""Seeded synthetic inputs for the Beam routed-MoE layer.

This module holds the layer shapes and the seeded random draws that feed both the CUDA
library and the CPU oracle. It holds none of the method's arithmetic: no routing, no
activation, no reduction. Every tensor is drawn from its own generator, seeded from
(seed, tensor tag), so two workloads that share a seed share their weights whatever their
token count.

Shapes come from the Beam release pages:
  * "Reflection releases Beam, a 501B open MoE model with 1M context", Architecture
    paragraph: hidden size 5,120; 256 experts per MoE layer in 8 groups of 32; the 4 best
    groups are kept; 8 experts per token; SwiGLU experts of intermediate size 2,560;
    outputs scaled by 2.5.
  * transformers "Beam" model doc, Overview, "Sparse MoE" bullet: the config names
    n_group, topk_group and routed_scaling_factor.

Value distributions (the pages give none; these are the synthetic recipe):
  x ~ N(0, 1) rounded to BF16; router weight ~ N(0, 0.02^2) FP32; expert bias ~ U(-0.1, 0.1)
  FP32; gate/up ~ N(0, 1/d) and down ~ N(0, 1/I), both rounded to BF16 (std 1/sqrt(fan_in)).
  The skewed-load workload adds +0.5 to the bias of 16 seeded "hot" experts.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Shape of one routed-MoE layer (names follow the transformers BeamConfig fields)."""

    d: int = 5120            # hidden size
    I: int = 2560            # expert intermediate size
    E: int = 256             # routed experts
    n_group: int = 8         # expert groups
    topk_group: int = 4      # groups kept per token
    top_k: int = 8           # experts per token
    scale: float = 2.5       # routed_scaling_factor


BEAM = MoEShape()
TINY = MoEShape(d=512, I=256)

# Tags that decorrelate the per-tensor generators.
_TAG = {"x": 1, "router_w": 2, "bias": 3, "w_gate": 4, "w_up": 5, "w_down": 6, "hot": 7, "sample": 8}


def generator(seed: int, tag: str, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _TAG[tag])
    return g


def make_tokens(shape: MoEShape, T: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """x [T, d] BF16, N(0, 1)."""
    g = generator(seed, "x", device)
    return torch.randn((T, shape.d), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_router(shape: MoEShape, seed: int = 0, device="cpu", hot_experts: int = 0, hot_bias: float = 0.5):
    """Router weight [E, d] FP32 ~ N(0, 0.02^2) and expert bias [E] FP32 ~ U(-0.1, 0.1).

    With hot_experts > 0, that many experts (a seeded permutation's first entries) get
    +hot_bias on top of their bias, which skews the per-expert load.
    """
    g = generator(seed, "router_w", device)
    w = torch.randn((shape.E, shape.d), generator=g, device=device, dtype=torch.float32).mul_(0.02)
    gb = generator(seed, "bias", device)
    b = torch.rand((shape.E,), generator=gb, device=device, dtype=torch.float32).mul_(0.2).sub_(0.1)
    if hot_experts:
        hot = hot_expert_ids(shape, hot_experts, seed)
        b[hot.to(device)] += hot_bias
    return w, b


def hot_expert_ids(shape: MoEShape, n: int, seed: int = 0) -> torch.Tensor:
    g = generator(seed, "hot", "cpu")
    return torch.randperm(shape.E, generator=g)[:n]


# Experts drawn together per generator call: as many as fit this many FP32 bytes (all 256
# Tiny experts in one draw; ten Beam experts).
_DRAW_BYTES = 1 << 29


def _expert_chunks(E: int, rows: int, fan_in: int):
    n = max(1, min(E, _DRAW_BYTES // (rows * fan_in * 4)))
    return [(e0, min(E, e0 + n)) for e0 in range(0, E, n)]


def make_experts(shape: MoEShape, seed: int = 0, device="cpu"):
    """w_gate, w_up [E, I, d] and w_down [E, d, I], BF16, std 1/sqrt(fan_in).

    Drawn in FP32 a few experts at a time (at most 512 MB of FP32 per draw), scaled, then
    rounded to BF16: a handful of launches at the Tiny shape, bounded extra memory at
    Beam's.
    """
    E, d, I = shape.E, shape.d, shape.I
    out = []
    for tag, rows, fan_in in (("w_gate", I, d), ("w_up", I, d), ("w_down", d, I)):
        g = generator(seed, tag, device)
        w = torch.empty((E, rows, fan_in), device=device, dtype=torch.bfloat16)
        std = 1.0 / math.sqrt(fan_in)
        for e0, e1 in _expert_chunks(E, rows, fan_in):
            w[e0:e1].copy_(torch.randn((e1 - e0, rows, fan_in), generator=g, device=device,
                                       dtype=torch.float32).mul_(std))
        out.append(w)
    return tuple(out)


FP8_MAX = 448.0  # largest finite FP8 E4M3 value


def quantize_rows_fp8(w: torch.Tensor):
    """Weight-only FP8 checkpoint recipe (the pages ship FP8 checkpoints but give no recipe;
    this is the plainest per-row one): per output row r, scale[r] = max|w[r]| / 448 (FP32)
    and q[r] = w[r] / scale[r] rounded to E4M3 by torch. Returns (q as uint8, scale)."""
    wf = w.float()
    scale = wf.abs().amax(dim=-1).clamp_min(1e-30) / FP8_MAX
    q = (wf / scale.unsqueeze(-1)).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale


def make_experts_fp8(shape: MoEShape, seed: int = 0, device="cpu"):
    """The experts of make_experts (same draws), quantised per row with quantize_rows_fp8:
    ((wg_q, wg_scale), (wu_q, wu_scale), (wd_q, wd_scale)) with q uint8 [E, rows, cols] and
    scale float32 [E, rows]. Drawn in the same chunks as make_experts."""
    E, d, I = shape.E, shape.d, shape.I
    out = []
    for tag, rows, fan_in in (("w_gate", I, d), ("w_up", I, d), ("w_down", d, I)):
        g = generator(seed, tag, device)
        q = torch.empty((E, rows, fan_in), device=device, dtype=torch.uint8)
        sc = torch.empty((E, rows), device=device, dtype=torch.float32)
        std = 1.0 / math.sqrt(fan_in)
        for e0, e1 in _expert_chunks(E, rows, fan_in):
            w = torch.randn((e1 - e0, rows, fan_in), generator=g, device=device, dtype=torch.float32).mul_(std)
            q[e0:e1], sc[e0:e1] = quantize_rows_fp8(w.to(torch.bfloat16))
        out.append((q, sc))
    return tuple(out)


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)  # FP4 E2M1 codes 0..7


def quantize_nvfp4(w: torch.Tensor):
    """NVFP4 checkpoint recipe for weight matrices w [..., rows, cols] (cols a multiple of
    16); the pages name the format but give no recipe, this is the plainest public one:
    one FP32 tensor scale per matrix t = max|w| / (448 * 6); per block of 16 consecutive
    elements of a row, an E4M3 scale bs = (block max|w|) / 6 / t rounded to E4M3 by torch;
    codes = the E2M1 magnitude nearest to |w| / (t * bs) (ties to the smaller), bit 3 the
    sign, packed two per byte (element 2k in the low half of byte k). Returns (codes uint8
    [..., rows, cols/2], block scales as E4M3 codes uint8 [..., rows, cols/16], t float32
    [...])."""
    wf = w.float()
    *lead, rows, cols = wf.shape
    t = (wf.abs().amax(dim=(-2, -1)) / (448.0 * 6.0)).clamp_min(1e-30)
    blocks = wf.reshape(*lead, rows, cols // 16, 16)
    bs = (blocks.abs().amax(dim=-1) / 6.0 / t[..., None, None]).to(torch.float8_e4m3fn)
    denom = (t[..., None, None] * bs.float()).unsqueeze(-1)
    v = torch.where(denom > 0, blocks / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(blocks))
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], device=w.device)
    mag = torch.bucketize(v.abs().contiguous(), mids)                      # 0..7
    code = (mag | ((v < 0) & (mag > 0)).to(mag.dtype) << 3).to(torch.uint8).reshape(*lead, rows, cols)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), bs.view(torch.uint8).contiguous(), t.float()


def make_experts_nvfp4(shape: MoEShape, seed: int = 0, device="cpu"):
    """The experts of make_experts (same draws), quantised with quantize_nvfp4, one tensor
    scale per expert matrix: ((wg_q, wg_bs, wg_t), (wu_q, wu_bs, wu_t), (wd_q, wd_bs, wd_t))
    with codes uint8 [E, rows, cols/2], block scales uint8 [E, rows, cols/16], t float32 [E]."""
    E, d, I = shape.E, shape.d, shape.I
    out = []
    for tag, rows, fan_in in (("w_gate", I, d), ("w_up", I, d), ("w_down", d, I)):
        g = generator(seed, tag, device)
        q = torch.empty((E, rows, fan_in // 2), device=device, dtype=torch.uint8)
        bs = torch.empty((E, rows, fan_in // 16), device=device, dtype=torch.uint8)
        t = torch.empty((E,), device=device, dtype=torch.float32)
        std = 1.0 / math.sqrt(fan_in)
        for e0, e1 in _expert_chunks(E, rows, fan_in):
            w = torch.randn((e1 - e0, rows, fan_in), generator=g, device=device, dtype=torch.float32).mul_(std)
            q[e0:e1], bs[e0:e1], t[e0:e1] = quantize_nvfp4(w.to(torch.bfloat16))
        out.append((q, bs, t))
    return tuple(out)


def sample_tokens(T: int, n: int, seed: int = 0) -> torch.Tensor:
    """A seeded, sorted subset of n distinct token indices out of T (all of them if n >= T)."""
    if n >= T:
        return torch.arange(T, dtype=torch.int64)
    g = generator(seed, "sample", "cpu")
    return torch.randperm(T, generator=g)[:n].sort().values


# The named workloads: (shape, T, hot experts).
WORKLOADS = {
    "tiny": (TINY, 128, 0),
    "decode": (BEAM, 16, 0),
    "prefill": (BEAM, 4096, 0),
    "skewed": (BEAM, 32768, 16),
}
SWEEP_T = (1, 8, 64, 256, 1024, 4096, 16384)
