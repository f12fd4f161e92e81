"""Tensor-level calls over the C ABI: allocate outputs, check shapes, call the library.

    out = moe.forward(x, router_w, bias, w_gate, w_up, w_down)          # Beam shape
    idx, w = moe.route(x, router_w, bias, shape=workloads.TINY)
    logits = moe.router_logits(x, router_w)
    out = moe.forward_host(x_pinned, ...)     # host in, host out, one library call
    part = moe.forward_shard(x, router_w, bias, wg[lo:hi], wu[lo:hi], wd[lo:hi], lo, hi)  # FP32
    x = moe.rmsnorm(stream, gamma, eps)
    new_stream = moe.sublayer_forward(stream, pre_gamma, post_gamma, eps, k, router_w, bias, w_gate, w_up, w_down)

All compute runs in libbeam_moe.so; nothing here touches the numbers.
"""
from __future__ import annotations

import torch

from . import abi
from .workloads import BEAM, MoEShape


def _check_inputs(shape: MoEShape, x, router_w, bias=None):
    T = x.shape[0]
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.shape == (T, shape.d) and x.is_contiguous()
    assert router_w.dtype == torch.float32 and router_w.shape == (shape.E, shape.d) and router_w.is_contiguous()
    if bias is not None:
        assert bias.dtype == torch.float32 and bias.shape == (shape.E,) and bias.is_contiguous()
    return T


def route(x, router_w, bias, shape: MoEShape = BEAM, stream=None):
    T = _check_inputs(shape, x, router_w, bias)
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device=x.device)
    abi.beam_moe_route_ex(shape, x, router_w, bias, T, idx, w, stream)
    return idx, w


def router_logits(x, router_w, shape: MoEShape = BEAM, stream=None):
    T = _check_inputs(shape, x, router_w)
    logits = torch.empty((T, shape.E), dtype=torch.float32, device=x.device)
    abi.beam_moe_router_logits(shape, x, router_w, T, logits, stream)
    return logits


def forward(x, router_w, bias, w_gate, w_up, w_down, shape: MoEShape = BEAM, out=None, stream=None):
    T = _check_inputs(shape, x, router_w, bias)
    for w, rows, cols in ((w_gate, shape.I, shape.d), (w_up, shape.I, shape.d), (w_down, shape.d, shape.I)):
        assert w.dtype == torch.bfloat16 and w.shape == (shape.E, rows, cols) and w.is_contiguous()
    if out is None:
        out = torch.empty((T, shape.d), dtype=torch.bfloat16, device=x.device)
    abi.beam_moe_forward_ex(shape, x, router_w, bias, w_gate, w_up, w_down, T, out, stream)
    return out


def forward_fp8(x, router_w, bias, experts_fp8, shape: MoEShape = BEAM, out=None, stream=None):
    """The block with FP8 E4M3 expert weights: experts_fp8 = ((wg_q, gs), (wu_q, us), (wd_q, ds))
    with codes uint8 [E, I, d], [E, I, d], [E, d, I] and FP32 row scales [E, I], [E, I], [E, d]
    (workloads.make_experts_fp8 builds them)."""
    T = _check_inputs(shape, x, router_w, bias)
    (wg, gs), (wu, us), (wd, ds) = experts_fp8
    for (w, sc), rows, cols in (((wg, gs), shape.I, shape.d), ((wu, us), shape.I, shape.d),
                                ((wd, ds), shape.d, shape.I)):
        assert w.dtype == torch.uint8 and w.shape == (shape.E, rows, cols) and w.is_contiguous()
        assert sc.dtype == torch.float32 and sc.shape == (shape.E, rows) and sc.is_contiguous()
    if out is None:
        out = torch.empty((T, shape.d), dtype=torch.bfloat16, device=x.device)
    abi.beam_moe_forward_fp8(shape, x, router_w, bias, wg, gs, wu, us, wd, ds, T, out, stream)
    return out


def forward_nvfp4(x, router_w, bias, experts_nvfp4, shape: MoEShape = BEAM, out=None, stream=None):
    """The block with NVFP4 expert weights: experts_nvfp4 = ((wg_q, wg_bs, wg_t), (wu_q, wu_bs, wu_t),
    (wd_q, wd_bs, wd_t)) with codes uint8 [E, rows, cols/2], E4M3 block scales uint8
    [E, rows, cols/16] and FP32 tensor scales [E] (workloads.make_experts_nvfp4 builds them)."""
    T = _check_inputs(shape, x, router_w, bias)
    parts = []
    for (q, bs, t), rows, cols in zip(experts_nvfp4, (shape.I, shape.I, shape.d), (shape.d, shape.d, shape.I)):
        assert q.dtype == torch.uint8 and q.shape == (shape.E, rows, cols // 2) and q.is_contiguous()
        assert bs.dtype == torch.uint8 and bs.shape == (shape.E, rows, cols // 16) and bs.is_contiguous()
        assert t.dtype == torch.float32 and t.shape == (shape.E,) and t.is_contiguous()
        parts += [q, bs, t]
    if out is None:
        out = torch.empty((T, shape.d), dtype=torch.bfloat16, device=x.device)
    abi.beam_moe_forward_nvfp4(shape, x, router_w, bias, *parts, T, out, stream)
    return out


def forward_host(x_host, router_w, bias, w_gate, w_up, w_down, shape: MoEShape = BEAM, out_host=None, stream=None):
    """Host tokens in, host output out, in one library call (beam_moe_forward_host): the copy
    of x to the device, the block and the copy of the output back, on `stream`; returns
    out_host once the stream has finished. Pinned host tensors keep the copies asynchronous."""
    T = x_host.shape[0]
    assert x_host.dtype == torch.bfloat16 and not x_host.is_cuda and x_host.shape == (T, shape.d)
    assert x_host.is_contiguous()
    for w, rows, cols in ((w_gate, shape.I, shape.d), (w_up, shape.I, shape.d), (w_down, shape.d, shape.I)):
        assert w.dtype == torch.bfloat16 and w.shape == (shape.E, rows, cols) and w.is_contiguous()
    if out_host is None:
        out_host = torch.empty((T, shape.d), dtype=torch.bfloat16, pin_memory=True)
    assert out_host.dtype == torch.bfloat16 and not out_host.is_cuda and out_host.shape == (T, shape.d)
    abi.beam_moe_forward_host(shape, x_host, router_w, bias, w_gate, w_up, w_down, T, out_host, stream)
    return out_host


def rmsnorm(v, gamma, eps: float, out=None, stream=None):
    """RMSNorm of the rows of a BF16 [T, d] tensor with a BF16 gain [d]."""
    T, d = v.shape
    assert v.dtype == torch.bfloat16 and v.is_cuda and v.is_contiguous()
    assert gamma.dtype == torch.bfloat16 and gamma.shape == (d,) and gamma.is_contiguous()
    if out is None:
        out = torch.empty_like(v)
    abi.beam_moe_rmsnorm(d, v, gamma, eps, T, out, stream)
    return out


def sublayer_forward(stream_in, pre_gamma, post_gamma, eps: float, k: int, router_w, bias, w_gate, w_up, w_down,
                     shape: MoEShape = BEAM, out=None, stream=None):
    """The MoE sublayer on the residual stream: pre-norm, MoE block, post-norm and the
    depth-scaled residual for contribution k. out may be stream_in (in place)."""
    T = _check_inputs(shape, stream_in, router_w, bias)
    for g in (pre_gamma, post_gamma):
        assert g.dtype == torch.bfloat16 and g.shape == (shape.d,) and g.is_contiguous()
    for w, rows, cols in ((w_gate, shape.I, shape.d), (w_up, shape.I, shape.d), (w_down, shape.d, shape.I)):
        assert w.dtype == torch.bfloat16 and w.shape == (shape.E, rows, cols) and w.is_contiguous()
    if out is None:
        out = torch.empty_like(stream_in)
    abi.beam_moe_sublayer_forward(shape, stream_in, pre_gamma, post_gamma, eps, k, router_w, bias, w_gate, w_up,
                                  w_down, T, out, stream)
    return out


def forward_shard(x, router_w, bias, w_gate, w_up, w_down, e_begin: int, e_end: int, shape: MoEShape = BEAM,
                  out=None, stream=None):
    """One expert-parallel shard: this device's experts [e_begin, e_end) (w_* hold only
    those); returns the FP32 partial output over the slots routed to them. Summing the
    partials of shards covering every expert gives the block's output."""
    T = _check_inputs(shape, x, router_w, bias)
    n = e_end - e_begin
    for w, rows, cols in ((w_gate, shape.I, shape.d), (w_up, shape.I, shape.d), (w_down, shape.d, shape.I)):
        assert w.dtype == torch.bfloat16 and w.shape == (n, rows, cols) and w.is_contiguous()
    if out is None:
        out = torch.empty((T, shape.d), dtype=torch.float32, device=x.device)
    abi.beam_moe_forward_shard(shape, x, router_w, bias, w_gate, w_up, w_down, e_begin, e_end, T, out, stream)
    return out


def dense_mlp(x, w_gate, w_up, w_down, out=None, stream=None):
    """Dense SwiGLU MLP on BF16 [T, d] tokens with weights [I, d], [I, d], [d, I]."""
    T, d = x.shape
    I = w_gate.shape[0]
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    for w, shp in ((w_gate, (I, d)), (w_up, (I, d)), (w_down, (d, I))):
        assert w.dtype == torch.bfloat16 and tuple(w.shape) == shp and w.is_contiguous()
    if out is None:
        out = torch.empty_like(x)
    abi.beam_moe_dense_mlp(d, I, x, w_gate, w_up, w_down, T, out, stream)
    return out


class ForwardGraph:
    """beam_moe_forward captured once in a CUDA graph for fixed device buffers and replayed:
    one graph launch instead of the call's kernel launches and scratch allocation. Write
    new tokens into `x` (same shape) before each replay; the result lands in `out`. The
    weights, router and bias must stay at the same addresses."""

    def __init__(self, x, router_w, bias, w_gate, w_up, w_down, shape: MoEShape = BEAM, out=None):
        self.x = x
        self.out = out if out is not None else torch.empty((x.shape[0], shape.d), dtype=torch.bfloat16,
                                                           device=x.device)
        args = (router_w, bias, w_gate, w_up, w_down, shape)
        side = torch.cuda.Stream(device=x.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # the library's per-device state and pool exist before capture
            forward(self.x, *args, out=self.out, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            forward(self.x, *args, out=self.out, stream=torch.cuda.current_stream())

    def replay(self):
        self.graph.replay()
        return self.out

