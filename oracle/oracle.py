"""ctypes front end of the plain-C CPU oracle (beam_moe_oracle.c).

TEST INFRASTRUCTURE ONLY: the test-suite, the package's smoke check and the benchmark's
CPU-baseline leg use this module; the CUDA library never does. The oracle shares no code
with the library; the only thing both sides share is the seeded input generator.

Arrays cross as numpy arrays: BF16 tensors as their uint16 bit patterns, FP32 as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "beam_moe_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libbeam_moe_oracle.so")
CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_default = None


class OracleCfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int), ("n_group", ctypes.c_int),
                ("topk_group", ctypes.c_int), ("top_k", ctypes.c_int), ("scale", ctypes.c_double)]


def cfg_of(shape) -> OracleCfg:
    """Accepts any object with the MoE shape fields (d, I, E, n_group, topk_group, top_k, scale)."""
    return OracleCfg(shape.d, shape.I, shape.E, shape.n_group, shape.topk_group, shape.top_k, float(shape.scale))


def _compile(src_path: str, out_path: str) -> str:
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src_path, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (skipped when up to date)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        _compile(SRC, LIB)
    return LIB


def build_variant(source_text: str, tag: str) -> str:
    """Compile a modified copy of the oracle source (used to show that the pins catch
    planted mistakes); returns the path of the shared library."""
    src = os.path.join(BUILD_DIR, f"variant_{tag}.c")
    os.makedirs(BUILD_DIR, exist_ok=True)
    with open(src, "w") as f:
        f.write(source_text)
    return _compile(src, os.path.join(BUILD_DIR, f"libvariant_{tag}.so"))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


class Oracle:
    """One loaded build of the oracle."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        cfgp = ctypes.POINTER(OracleCfg)
        L.oracle_check_cfg.argtypes = [cfgp]
        L.oracle_router_logits.argtypes = [cfgp, P, P, i64, P]
        L.oracle_route.argtypes = [cfgp, P, P, i64, P, P, P, P, P, P, P]
        L.oracle_expert.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P]
        L.oracle_forward.argtypes = [cfgp, P, i64, P, i64, P, P, P, P, P, P, P, P, P, P]
        for f in (L.oracle_check_cfg, L.oracle_router_logits, L.oracle_route, L.oracle_expert, L.oracle_forward):
            f.restype = ctypes.c_int
        self.L = L
        self.path = path

    def check_cfg(self, shape) -> bool:
        cfg = cfg_of(shape)
        return self.L.oracle_check_cfg(ctypes.byref(cfg)) == 0

    def router_logits(self, shape, x_bits, router_w) -> np.ndarray:
        """FP32 logits [T, E] (FP64 sums rounded once)."""
        x_bits = _u16(x_bits)
        router_w = _f32(router_w)
        T = x_bits.shape[0]
        out = np.empty((T, shape.E), np.float32)
        cfg = cfg_of(shape)
        _check(self.L.oracle_router_logits(ctypes.byref(cfg), _ptr(x_bits), _ptr(router_w), T, _ptr(out)),
               "router_logits")
        return out

    def route(self, shape, logits, bias, debug: bool = False):
        """Routing from FP32 logits. Returns (idx [T,K] int32, w [T,K] float32) and, with
        debug=True, also a dict with s, c [T,E], gs [T,G], groups [T,TG], w64 [T,K]."""
        logits = _f32(logits)
        bias = _f32(bias)
        T = logits.shape[0]
        K, E, G, TG = shape.top_k, shape.E, shape.n_group, shape.topk_group
        idx = np.empty((T, K), np.int32)
        w = np.empty((T, K), np.float32)
        dbg = None
        if debug:
            dbg = dict(s=np.empty((T, E), np.float32), c=np.empty((T, E), np.float32),
                       gs=np.empty((T, G), np.float32), groups=np.empty((T, TG), np.int32),
                       w64=np.empty((T, K), np.float64))
        cfg = cfg_of(shape)
        extra = [_ptr(dbg[k]) if dbg else None for k in ("s", "c", "gs", "groups", "w64")]
        _check(self.L.oracle_route(ctypes.byref(cfg), _ptr(logits), _ptr(bias), T, _ptr(idx), _ptr(w), *extra),
               "route")
        return (idx, w, dbg) if debug else (idx, w)

    def expert(self, shape, x_row, wg_e, wu_e, wd_e) -> np.ndarray:
        """One SwiGLU expert on one FP64 row: returns y [d] FP64."""
        x_row = np.ascontiguousarray(x_row, dtype=np.float64)
        y = np.empty(shape.d, np.float64)
        _check(self.L.oracle_expert(shape.d, shape.I, _ptr(x_row), _ptr(_u16(wg_e)), _ptr(_u16(wu_e)),
                                    _ptr(_u16(wd_e)), _ptr(y)), "expert")
        return y

    def forward(self, shape, x_bits, bias, experts, tokens=None, router_w=None, logits=None, idx_in=None):
        """The MoE block for selected tokens (all if tokens is None).

        experts: a callable e -> (wg_e, wu_e, wd_e) uint16 arrays, or None for an expert
        that is not available (the oracle fails if a routed token needs it). It is called
        for every e in [0, E).
        Returns (out [n, d] FP64, idx [n, K] int32, w [n, K] float32).
        """
        x_bits = _u16(x_bits)
        bias = _f32(bias)
        T = x_bits.shape[0]
        tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
        n = T if tok is None else tok.shape[0]
        K, E = shape.top_k, shape.E
        keep = []
        arrs = [(ctypes.c_void_p * E)() for _ in range(3)]
        for e in range(E):
            ws = experts(e)
            if ws is None:
                continue
            for a, w in zip(arrs, ws):
                w = _u16(w)
                keep.append(w)
                a[e] = w.ctypes.data
        out = np.empty((n, shape.d), np.float64)
        idx = np.empty((n, K), np.int32)
        w = np.empty((n, K), np.float32)
        lg = None if logits is None else _f32(logits)
        rw = None if router_w is None else _f32(router_w)
        ii = None if idx_in is None else np.ascontiguousarray(idx_in, dtype=np.int32)
        cfg = cfg_of(shape)
        rc = self.L.oracle_forward(ctypes.byref(cfg), _ptr(x_bits), T, _ptr(tok), n, _ptr(lg), _ptr(rw), _ptr(bias),
                                   _ptr(ii), arrs[0], arrs[1], arrs[2], _ptr(out), _ptr(idx), _ptr(w))
        _check(rc, "forward")
        return out, idx, w


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def router_logits(*a, **k):
    return default().router_logits(*a, **k)


def route(*a, **k):
    return default().route(*a, **k)


def expert(*a, **k):
    return default().expert(*a, **k)


def forward(*a, **k):
    return default().forward(*a, **k)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a BF16 torch tensor (on any device)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def experts_from(wg, wu, wd, only=None):
    """An `experts` callable over host BF16 tensors [E, ...]; `only` (a set) limits which
    experts are handed to the oracle."""
    def get(e):
        if only is not None and e not in only:
            return None
        return bf16_bits(wg[e]), bf16_bits(wu[e]), bf16_bits(wd[e])
    return get
