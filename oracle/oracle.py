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
        L.oracle_rmsnorm.argtypes = [ctypes.c_int, P, P, ctypes.c_double, P]
        L.oracle_e4m3_decode.argtypes = [i64, P, P]
        L.oracle_expert_fp8.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P]
        L.oracle_residual.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P]
        dbl = ctypes.c_double
        L.oracle_e2m1_decode.argtypes = [i64, P, P]
        L.oracle_expert_nvfp4.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, dbl, P, P, dbl, P, P, dbl, P]
        L.oracle_round_bf16.argtypes = [i64, P, P]
        for f in (L.oracle_check_cfg, L.oracle_router_logits, L.oracle_route, L.oracle_expert, L.oracle_forward,
                  L.oracle_rmsnorm, L.oracle_residual, L.oracle_round_bf16, L.oracle_e4m3_decode,
                  L.oracle_expert_fp8, L.oracle_e2m1_decode, L.oracle_expert_nvfp4):
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


    def rmsnorm(self, v, gamma_bits, eps) -> np.ndarray:
        """RMSNorm of one FP64 row with a BF16 gain (bit patterns): FP64 result."""
        v = np.ascontiguousarray(v, dtype=np.float64)
        g = _u16(gamma_bits)
        assert g.shape == v.shape
        y = np.empty_like(v)
        _check(self.L.oracle_rmsnorm(v.shape[0], _ptr(v), _ptr(g), float(eps), _ptr(y)), "rmsnorm")
        return y

    def residual(self, stream, sub, k) -> np.ndarray:
        """Depth-scaled residual update for contribution k (>= 2): FP64 row."""
        stream = np.ascontiguousarray(stream, dtype=np.float64)
        sub = np.ascontiguousarray(sub, dtype=np.float64)
        out = np.empty_like(stream)
        _check(self.L.oracle_residual(stream.shape[0], int(k), _ptr(stream), _ptr(sub), _ptr(out)), "residual")
        return out

    def round_bf16(self, v) -> np.ndarray:
        """BF16 bit patterns nearest to FP64 values (same shape)."""
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, np.uint16)
        _check(self.L.oracle_round_bf16(v.size, _ptr(v), _ptr(out)), "round_bf16")
        return out

    def sublayer(self, shape, stream_bits, pre_gamma_bits, post_gamma_bits, eps, k, bias, experts, tokens,
                 x_bits=None, logits=None, router_w=None, idx_in=None, grouped=False):
        """The MoE sublayer for the rows `tokens` of a BF16 stream [T, d] (bit patterns),
        in the pages' order: x = RMSNorm_pre(stream) rounded to BF16 (the block's input
        hidden state), m = MoE(x), out = sqrt((k-1)/k) stream + RMSNorm_post(m) / sqrt(k).
        x_bits [T, d], if given, replaces the oracle's own rounded pre-norm output (so the
        rest can be checked given another implementation's BF16 input); logits / idx_in as
        in forward(). grouped: the MoE block through forward_grouped (for large token
        samples). Returns (out [n, d] FP64, x_rows [n, d] FP64 pre-norm before rounding)."""
        stream_bits = _u16(stream_bits)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        T, d = stream_bits.shape
        s64 = stream_bits[tokens].astype(np.uint32) << 16
        s64 = s64.view(np.float32).astype(np.float64)
        x_rows = np.stack([self.rmsnorm(s64[i], pre_gamma_bits, eps) for i in range(len(tokens))]) \
            if len(tokens) else np.zeros((0, d))
        if x_bits is None:
            x_bits = np.zeros((T, d), np.uint16)
            x_bits[tokens] = self.round_bf16(x_rows)
        if grouped:
            m, _ = self.forward_grouped(shape, x_bits, bias, experts, tokens, logits=logits, router_w=router_w,
                                        idx_in=idx_in)
        else:
            m, _, _ = self.forward(shape, x_bits, bias, experts, tokens=tokens, router_w=router_w, logits=logits,
                                   idx_in=idx_in)
        out = np.stack([self.residual(s64[i], self.rmsnorm(m[i], post_gamma_bits, eps), k)
                        for i in range(len(tokens))]) if len(tokens) else np.zeros((0, d))
        return out, x_rows


    def e4m3_decode(self, q) -> np.ndarray:
        """FP64 values of FP8 E4M3 codes (uint8 array, any shape)."""
        q = np.ascontiguousarray(q, dtype=np.uint8)
        out = np.empty(q.shape, np.float64)
        _check(self.L.oracle_e4m3_decode(q.size, _ptr(q), _ptr(out)), "e4m3_decode")
        return out

    def expert_fp8(self, shape, x_row, wg_q, gs, wu_q, us, wd_q, ds) -> np.ndarray:
        """One SwiGLU expert with FP8 E4M3 weights and per-row FP32 scales on one FP64 row."""
        x_row = np.ascontiguousarray(x_row, dtype=np.float64)
        arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (wg_q, wu_q, wd_q)]
        scs = [_f32(a) for a in (gs, us, ds)]
        y = np.empty(shape.d, np.float64)
        _check(self.L.oracle_expert_fp8(shape.d, shape.I, _ptr(x_row), _ptr(arrs[0]), _ptr(scs[0]), _ptr(arrs[1]),
                                        _ptr(scs[1]), _ptr(arrs[2]), _ptr(scs[2]), _ptr(y)), "expert_fp8")
        return y

    def e2m1_decode(self, codes) -> np.ndarray:
        """FP64 values of E2M1 (FP4) codes, one per byte (low 4 bits), any shape."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, np.float64)
        _check(self.L.oracle_e2m1_decode(c.size, _ptr(c), _ptr(out)), "e2m1_decode")
        return out

    def expert_nvfp4(self, shape, x_row, gate, up, down) -> np.ndarray:
        """One SwiGLU expert with NVFP4 weights on one FP64 row. gate, up, down are (codes,
        block scales, tensor scale): codes uint8 [rows, cols/2] (two per byte, element 2k in
        the low half), block scales E4M3 codes uint8 [rows, cols/16], tensor scale a float."""
        x_row = np.ascontiguousarray(x_row, dtype=np.float64)
        keep = [np.ascontiguousarray(a, dtype=np.uint8) for g in (gate, up, down) for a in g[:2]]
        ptrs = [_ptr(k) for k in keep]
        y = np.empty(shape.d, np.float64)
        _check(self.L.oracle_expert_nvfp4(shape.d, shape.I, _ptr(x_row), ptrs[0], ptrs[1], float(gate[2]), ptrs[2],
                                          ptrs[3], float(up[2]), ptrs[4], ptrs[5], float(down[2]), _ptr(y)),
               "expert_nvfp4")
        return y

    def _forward_with(self, shape, x_bits, bias, expert_of, tokens, logits=None, router_w=None, idx_in=None):
        """The MoE block for the rows `tokens` with the expert evaluated by expert_of(x_row, e)
        (an FP64 row in, an FP64 row out): the same routing as forward() (from `logits` if
        given), weights from the oracle's own sigmoid scores, weighted sum in FP64 in slot
        order. idx_in replaces the selection for the given rows."""
        x_bits = _u16(x_bits)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        lg = _f32(logits)[tokens] if logits is not None else self.router_logits(shape, x_bits[tokens], router_w)
        idx, _, dbg = self.route(shape, lg, bias, debug=True)
        w64 = dbg["w64"]
        if idx_in is not None:
            idx = np.asarray(idx_in, np.int32)
            s = dbg["s"].astype(np.float64)
            picked = np.take_along_axis(s, idx.astype(np.int64), axis=1)
            w64 = shape.scale * picked / picked.sum(axis=1, keepdims=True)
        out = np.zeros((len(tokens), shape.d), np.float64)
        for n, t in enumerate(tokens):
            xr = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            for k in range(shape.top_k):
                out[n] += w64[n, k] * expert_of(xr, int(idx[n, k]))
        return out, idx

    def forward_fp8(self, shape, x_bits, bias, experts_q, tokens, logits=None, router_w=None, idx_in=None):
        """The MoE block with FP8 experts for the rows `tokens` (composition of _forward_with),
        experts evaluated by expert_fp8. experts_q: e -> (wg_q, gs, wu_q, us, wd_q, ds)."""
        return self._forward_with(shape, x_bits, bias, lambda xr, e: self.expert_fp8(shape, xr, *experts_q(e)),
                                  tokens, logits=logits, router_w=router_w, idx_in=idx_in)

    def forward_nvfp4(self, shape, x_bits, bias, experts_q, tokens, logits=None, router_w=None, idx_in=None):
        """The MoE block with NVFP4 experts for the rows `tokens` (composition of
        _forward_with), experts evaluated by expert_nvfp4. experts_q: e -> (gate, up, down),
        each (codes, block scales, tensor scale) as expert_nvfp4 takes them."""
        return self._forward_with(shape, x_bits, bias, lambda xr, e: self.expert_nvfp4(shape, xr, *experts_q(e)),
                                  tokens, logits=logits, router_w=router_w, idx_in=idx_in)

    def forward_grouped(self, shape, x_bits, bias, experts, tokens, logits=None, router_w=None, idx_in=None):
        """forward() for many tokens at Beam size: the same routing (this oracle's, from
        `logits` if given), the same SwiGLU expert in FP64 with no intermediate rounding,
        the same FP64 sum over each token's slots in slot order, but each expert evaluated
        for all the tokens routed to it at once with numpy FP64 matrix products (a library
        matmul as the step; equal to forward() up to the order of FP64 additions inside
        the products). experts: callable e -> (wg_e, wu_e, wd_e) BF16 bit patterns.
        Returns (out [n, d] FP64, idx [n, K] int32)."""
        x_bits = _u16(x_bits)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        lg = _f32(logits)[tokens] if logits is not None else self.router_logits(shape, x_bits[tokens], router_w)
        idx, _, dbg = self.route(shape, lg, bias, debug=True)
        w64 = dbg["w64"]
        if idx_in is not None:
            idx = np.asarray(idx_in, np.int32)
            sc = dbg["s"].astype(np.float64)
            picked = np.take_along_axis(sc, idx.astype(np.int64), axis=1)
            w64 = shape.scale * picked / picked.sum(axis=1, keepdims=True)
        n, K = idx.shape
        xd = (x_bits[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        y = np.zeros((n, K, shape.d), np.float64)  # expert output of every (token, slot)
        for e in np.unique(idx):
            rows, slots = np.nonzero(idx == e)
            wg, wu, wd = (((_u16(a).astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
                          for a in experts(int(e)))
            xe = xd[rows]
            g = xe @ wg.T
            u = xe @ wu.T
            h = g / (1.0 + np.exp(-g)) * u
            y[rows, slots] = h @ wd.T
        out = np.zeros((n, shape.d), np.float64)
        for k in range(K):
            out += w64[:, k:k + 1] * y[:, k]
        return out, idx

    def forward_shard(self, shape, x_bits, bias, experts, e_begin, e_end, tokens, logits=None, router_w=None):
        """One expert-parallel shard's partial output for the rows `tokens`: the sum over the
        token's slots routed to experts [e_begin, e_end) of w_k * expert_k(x), FP64, with
        the oracle's own routing (from `logits` if given, else from router_w).
        experts: callable e -> (wg_e, wu_e, wd_e) bit patterns for the shard's experts."""
        x_bits = _u16(x_bits)
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        lg = _f32(logits)[tokens] if logits is not None else self.router_logits(shape, x_bits[tokens], router_w)
        idx, _, dbg = self.route(shape, lg, bias, debug=True)
        out = np.zeros((len(tokens), shape.d), np.float64)
        for n, t in enumerate(tokens):
            xr = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            for k in range(shape.top_k):
                e = int(idx[n, k])
                if e_begin <= e < e_end:
                    out[n] += dbg["w64"][n, k] * self.expert(shape, xr, *experts(e))
        return out


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


def rmsnorm(*a, **k):
    return default().rmsnorm(*a, **k)


def residual(*a, **k):
    return default().residual(*a, **k)


def round_bf16(*a, **k):
    return default().round_bf16(*a, **k)


def sublayer(*a, **k):
    return default().sublayer(*a, **k)


def forward_shard(*a, **k):
    return default().forward_shard(*a, **k)


def e4m3_decode(*a, **k):
    return default().e4m3_decode(*a, **k)


def expert_fp8(*a, **k):
    return default().expert_fp8(*a, **k)


def forward_grouped(*a, **k):
    return default().forward_grouped(*a, **k)


def forward_fp8(*a, **k):
    return default().forward_fp8(*a, **k)


def e2m1_decode(*a, **k):
    return default().e2m1_decode(*a, **k)


def expert_nvfp4(*a, **k):
    return default().expert_nvfp4(*a, **k)


def forward_nvfp4(*a, **k):
    return default().forward_nvfp4(*a, **k)


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
