"""Thin ctypes binding of libbeam_moe.so (include/beam_moe.h): same names, argument
marshalling only. Every step of the MoE forward pass runs in the library's CUDA kernels;
this module only turns torch tensors into device pointers and status codes into
exceptions. There is no fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbeam_moe.so")

BEAM_MOE_OK = 0
BEAM_MOE_ERR_ARG = -1
BEAM_MOE_ERR_ALIGN = -2
BEAM_MOE_ERR_CUDA = -3
BEAM_MOE_ERR_DEVICE = -4
BEAM_MOE_MAX_TOKENS = 262144
BEAM_MOE_NOALLOC_MAX_TOKENS = 8192
BEAM_MOE_NOALLOC_SCRATCH_BYTES = 40 << 20

STAGES = ("pre_norm", "router_split", "router_logits", "router_select", "dispatch_count", "dispatch_scan",
          "dispatch_scatter", "gather", "expert_mlp", "combine", "act_prep")

# Every symbol include/beam_moe.h declares.
EXPORTS = ("beam_moe_default_config", "beam_moe_route", "beam_moe_route_ex", "beam_moe_forward",
           "beam_moe_forward_ex", "beam_moe_router_logits", "beam_moe_last_error", "beam_moe_device_status",
           "beam_moe_timing_enable", "beam_moe_timing_read", "beam_moe_last_launch_count",
           "beam_moe_route_noalloc", "beam_moe_rmsnorm", "beam_moe_sublayer_forward", "beam_moe_forward_shard",
           "beam_moe_dense_mlp", "beam_moe_forward_fp8", "beam_moe_selftest_wait_timeout",
           "beam_moe_route_noalloc_plan", "beam_moe_route_noalloc_status", "beam_moe_route_noalloc_selftest",
           "beam_moe_forward_host", "beam_moe_debug_poison_scratch", "beam_moe_forward_nvfp4")


class BeamMoeConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int), ("n_group", ctypes.c_int),
                ("topk_group", ctypes.c_int), ("top_k", ctypes.c_int), ("scale", ctypes.c_float)]

    @classmethod
    def of(cls, shape) -> "BeamMoeConfig":
        return cls(shape.d, shape.I, shape.E, shape.n_group, shape.topk_group, shape.top_k, float(shape.scale))


_cfg_cache = {}


class BeamMoeError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"beam_moe error {code}: {message}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libbeam_moe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with python -m sparse_moe_transformer_bias_b300.build")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.c_void_p
            i = ctypes.c_int
            cfgp = ctypes.POINTER(BeamMoeConfig)
            L.beam_moe_default_config.restype = BeamMoeConfig
            L.beam_moe_default_config.argtypes = []
            L.beam_moe_route.argtypes = [P, P, P, i, P, P, P]
            L.beam_moe_route_ex.argtypes = [cfgp, P, P, P, i, P, P, P]
            L.beam_moe_forward.argtypes = [P, P, P, P, P, P, i, P, P]
            L.beam_moe_forward_ex.argtypes = [cfgp, P, P, P, P, P, P, i, P, P]
            L.beam_moe_router_logits.argtypes = [cfgp, P, P, i, P, P]
            L.beam_moe_forward_host.argtypes = [cfgp, P, P, P, P, P, P, i, P, P]
            L.beam_moe_route_noalloc.argtypes = [cfgp, P, P, P, i, P, P, P]
            L.beam_moe_route_noalloc_plan.argtypes = [cfgp, i, i, ctypes.POINTER(ctypes.c_int)]
            L.beam_moe_route_noalloc_status.argtypes = [P]
            L.beam_moe_route_noalloc_selftest.argtypes = [P]
            f32 = ctypes.c_float
            L.beam_moe_rmsnorm.argtypes = [i, P, P, f32, i, P, P]
            L.beam_moe_sublayer_forward.argtypes = [cfgp, P, P, P, f32, i, P, P, P, P, P, i, P, P]
            L.beam_moe_forward_shard.argtypes = [cfgp, P, P, P, P, P, P, i, i, i, P, P]
            L.beam_moe_dense_mlp.argtypes = [i, i, P, P, P, P, i, P, P]
            L.beam_moe_forward_fp8.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i, P, P]
            L.beam_moe_forward_nvfp4.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, i, P, P]
            L.beam_moe_selftest_wait_timeout.argtypes = [P]
            L.beam_moe_last_error.restype = ctypes.c_char_p
            L.beam_moe_last_error.argtypes = []
            L.beam_moe_device_status.argtypes = [P]
            L.beam_moe_timing_enable.argtypes = [i]
            L.beam_moe_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), i]
            L.beam_moe_last_launch_count.argtypes = []
            L.beam_moe_debug_poison_scratch.argtypes = [i]
            for f in ("beam_moe_route", "beam_moe_route_ex", "beam_moe_forward", "beam_moe_forward_ex",
                      "beam_moe_router_logits", "beam_moe_device_status", "beam_moe_timing_enable",
                      "beam_moe_timing_read", "beam_moe_last_launch_count", "beam_moe_route_noalloc",
                      "beam_moe_rmsnorm", "beam_moe_sublayer_forward", "beam_moe_forward_shard",
                      "beam_moe_dense_mlp", "beam_moe_forward_fp8", "beam_moe_selftest_wait_timeout",
           "beam_moe_route_noalloc_plan", "beam_moe_route_noalloc_status", "beam_moe_route_noalloc_selftest",
           "beam_moe_forward_host", "beam_moe_debug_poison_scratch", "beam_moe_forward_nvfp4"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(t):
    """Device pointer of a tensor (None/0 passes a null pointer, an int passes through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != BEAM_MOE_OK:
        raise BeamMoeError(rc, load().beam_moe_last_error().decode())
    return rc


def _cfg(cfg):
    if cfg is None:
        return None
    if isinstance(cfg, BeamMoeConfig):
        return ctypes.byref(cfg)
    c = _cfg_cache.get(cfg)  # shapes are frozen dataclasses: one struct per shape
    if c is None:
        c = _cfg_cache.setdefault(cfg, BeamMoeConfig.of(cfg))
    return ctypes.byref(c)


def beam_moe_default_config() -> BeamMoeConfig:
    return load().beam_moe_default_config()


def beam_moe_route(x, router_w, expert_bias, T, topk_idx, topk_w, stream=None):
    return _check(load().beam_moe_route(_ptr(x), _ptr(router_w), _ptr(expert_bias), int(T), _ptr(topk_idx),
                                        _ptr(topk_w), _stream(stream)))


def beam_moe_route_ex(cfg, x, router_w, expert_bias, T, topk_idx, topk_w, stream=None):
    return _check(load().beam_moe_route_ex(_cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), int(T),
                                           _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def beam_moe_forward(x, router_w, expert_bias, w_gate, w_up, w_down, T, out, stream=None):
    return _check(load().beam_moe_forward(_ptr(x), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate), _ptr(w_up),
                                          _ptr(w_down), int(T), _ptr(out), _stream(stream)))


def beam_moe_forward_ex(cfg, x, router_w, expert_bias, w_gate, w_up, w_down, T, out, stream=None):
    return _check(load().beam_moe_forward_ex(_cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate),
                                             _ptr(w_up), _ptr(w_down), int(T), _ptr(out), _stream(stream)))


def beam_moe_forward_host(cfg, x_host, router_w, expert_bias, w_gate, w_up, w_down, T, out_host, stream=None):
    """The block with x and out in host memory (pinned for asynchronous copies); returns once
    the stream has finished."""
    return _check(load().beam_moe_forward_host(_cfg(cfg), _ptr(x_host), _ptr(router_w), _ptr(expert_bias),
                                               _ptr(w_gate), _ptr(w_up), _ptr(w_down), int(T), _ptr(out_host),
                                               _stream(stream)))


def beam_moe_route_noalloc(cfg, x, router_w, expert_bias, T, topk_idx, topk_w, stream=None):
    """beam_moe_route_ex without any device allocation (fixed scratch array in the
    library; T <= BEAM_MOE_NOALLOC_MAX_TOKENS)."""
    return _check(load().beam_moe_route_noalloc(_cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), int(T),
                                                _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def beam_moe_route_noalloc_plan(cfg, T, num_sms) -> int:
    """K split planes a no-allocation router call with T tokens makes on a GPU with num_sms
    SMs (host-only query; raises if the batch does not fit the fixed array)."""
    n = ctypes.c_int(0)
    _check(load().beam_moe_route_noalloc_plan(_cfg(cfg), int(T), int(num_sms), ctypes.byref(n)))
    return n.value


def beam_moe_route_noalloc_status(stream=None):
    """Raise if a kernel of the no-allocation router recorded an error (read and clear)."""
    return _check(load().beam_moe_route_noalloc_status(_stream(stream)))


def beam_moe_route_noalloc_selftest(stream=None):
    """Queue the no-allocation router's failure-detection self-test (a bounded wait that
    runs out); read the outcome with beam_moe_route_noalloc_status()."""
    return _check(load().beam_moe_route_noalloc_selftest(_stream(stream)))


def beam_moe_forward_shard(cfg, x, router_w, expert_bias, w_gate, w_up, w_down, e_begin, e_end, T, out_partial,
                           stream=None):
    return _check(load().beam_moe_forward_shard(_cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate),
                                                _ptr(w_up), _ptr(w_down), int(e_begin), int(e_end), int(T),
                                                _ptr(out_partial), _stream(stream)))


def beam_moe_forward_fp8(cfg, x, router_w, expert_bias, w_gate_q, gate_scale, w_up_q, up_scale, w_down_q, down_scale,
                         T, out, stream=None):
    return _check(load().beam_moe_forward_fp8(_cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate_q),
                                              _ptr(gate_scale), _ptr(w_up_q), _ptr(up_scale), _ptr(w_down_q),
                                              _ptr(down_scale), int(T), _ptr(out), _stream(stream)))


def beam_moe_forward_nvfp4(cfg, x, router_w, expert_bias, w_gate_q, gate_block_scale, gate_tensor_scale, w_up_q,
                           up_block_scale, up_tensor_scale, w_down_q, down_block_scale, down_tensor_scale, T, out,
                           stream=None):
    return _check(load().beam_moe_forward_nvfp4(
        _cfg(cfg), _ptr(x), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate_q), _ptr(gate_block_scale),
        _ptr(gate_tensor_scale), _ptr(w_up_q), _ptr(up_block_scale), _ptr(up_tensor_scale), _ptr(w_down_q),
        _ptr(down_block_scale), _ptr(down_tensor_scale), int(T), _ptr(out), _stream(stream)))


def beam_moe_selftest_wait_timeout(stream=None):
    """Queue the failure-detection self-test (a bounded wait that runs out); read the
    outcome with beam_moe_device_status()."""
    return _check(load().beam_moe_selftest_wait_timeout(_stream(stream)))


def beam_moe_dense_mlp(d, I, x, w_gate, w_up, w_down, T, out, stream=None):
    return _check(load().beam_moe_dense_mlp(int(d), int(I), _ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), int(T),
                                            _ptr(out), _stream(stream)))


def beam_moe_rmsnorm(d, v, gamma, eps, T, out, stream=None):
    return _check(load().beam_moe_rmsnorm(int(d), _ptr(v), _ptr(gamma), float(eps), int(T), _ptr(out),
                                          _stream(stream)))


def beam_moe_sublayer_forward(cfg, stream_in, pre_gamma, post_gamma, eps, k, router_w, expert_bias, w_gate, w_up,
                              w_down, T, stream_out, stream=None):
    return _check(load().beam_moe_sublayer_forward(_cfg(cfg), _ptr(stream_in), _ptr(pre_gamma), _ptr(post_gamma),
                                                   float(eps), int(k), _ptr(router_w), _ptr(expert_bias),
                                                   _ptr(w_gate), _ptr(w_up), _ptr(w_down), int(T), _ptr(stream_out),
                                                   _stream(stream)))


def beam_moe_router_logits(cfg, x, router_w, T, logits, stream=None):
    return _check(load().beam_moe_router_logits(_cfg(cfg), _ptr(x), _ptr(router_w), int(T), _ptr(logits),
                                                _stream(stream)))


def beam_moe_last_error() -> str:
    return load().beam_moe_last_error().decode()


def beam_moe_device_status(stream=None):
    return _check(load().beam_moe_device_status(_stream(stream)))


def beam_moe_timing_enable(enable: bool):
    return _check(load().beam_moe_timing_enable(1 if enable else 0))


def beam_moe_timing_read() -> dict:
    buf = (ctypes.c_float * len(STAGES))()
    n = load().beam_moe_timing_read(buf, len(STAGES))
    if n < 0:
        _check(n)
    return {name: float(buf[i]) for i, name in enumerate(STAGES)}


def beam_moe_debug_poison_scratch(enable: bool):
    """Fill every scratch allocation with NaN bytes before use (debug aid, process-wide)."""
    return _check(load().beam_moe_debug_poison_scratch(1 if enable else 0))


def beam_moe_last_launch_count() -> int:
    return int(load().beam_moe_last_launch_count())
