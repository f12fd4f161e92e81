"""The C-ABI library loads, exports every declared symbol and rejects bad arguments on
the host (no GPU needed: every call here fails or returns before touching the device)."""
import ctypes
import os
import re

import pytest

from sparse_moe_transformer_bias_b300 import abi, build, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BEAM_MOE_API\s+[\w\s\*]*?\b(beam_moe_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(abi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_default_config_is_beam(lib):
    c = abi.beam_moe_default_config()
    assert (c.d, c.I, c.E, c.n_group, c.topk_group, c.top_k, c.scale) == (5120, 2560, 256, 8, 4, 8, 2.5)


FAKE = 1 << 20  # 16-byte aligned, never dereferenced by argument checks


def call_forward(cfg, T=4, x=FAKE, wr=FAKE, b=FAKE, wg=FAKE, wu=FAKE, wd=FAKE, out=FAKE):
    return lib_().beam_moe_forward_ex(ctypes.byref(cfg), x, wr, b, wg, wu, wd, T, out, None)


def lib_():
    return abi.load()


def cfg_of(**kw):
    base = dict(d=5120, I=2560, E=256, n_group=8, topk_group=4, top_k=8, scale=2.5)
    base.update(kw)
    return abi.BeamMoeConfig(**base)


@pytest.mark.parametrize("kw,what", [
    (dict(d=5000), "d=5000"), (dict(I=100), "I=100"), (dict(E=250), "E=250"), (dict(n_group=9, E=288), "n_group"),
    (dict(topk_group=9), "topk_group"), (dict(topk_group=0), "topk_group"), (dict(top_k=0), "top_k"),
    (dict(top_k=33), "top_k"), (dict(scale=float("inf")), "scale"),
])
def test_bad_config_rejected(lib, kw, what):
    assert call_forward(cfg_of(**kw)) == abi.BEAM_MOE_ERR_ARG
    assert what.split("=")[0] in abi.beam_moe_last_error()


def test_bad_token_count_rejected(lib):
    assert call_forward(cfg_of(), T=-1) == abi.BEAM_MOE_ERR_ARG
    assert call_forward(cfg_of(), T=abi.BEAM_MOE_MAX_TOKENS + 1) == abi.BEAM_MOE_ERR_ARG


@pytest.mark.parametrize("arg", ["x", "wr", "b", "wg", "wu", "wd", "out"])
def test_null_and_misaligned_pointers_rejected(lib, arg):
    assert call_forward(cfg_of(), **{arg: None}) == abi.BEAM_MOE_ERR_ARG
    assert "null" in abi.beam_moe_last_error()
    assert call_forward(cfg_of(), **{arg: FAKE + 8}) == abi.BEAM_MOE_ERR_ALIGN
    assert "aligned" in abi.beam_moe_last_error()


def test_zero_tokens_is_a_no_op(lib):
    assert call_forward(cfg_of(), T=0) == abi.BEAM_MOE_OK
    assert lib.beam_moe_route_ex(ctypes.byref(cfg_of(**dict(d=512, I=256))), FAKE, FAKE, FAKE, 0, FAKE, FAKE,
                                 None) == abi.BEAM_MOE_OK
    assert lib.beam_moe_router_logits(ctypes.byref(cfg_of()), FAKE, FAKE, 0, FAKE, None) == abi.BEAM_MOE_OK
    assert abi.beam_moe_last_launch_count() == 0


def test_binding_raises_with_message(lib):
    with pytest.raises(abi.BeamMoeError, match="T=-3"):
        abi.beam_moe_route_ex(W.TINY, FAKE, FAKE, FAKE, -3, FAKE, FAKE, stream=0)


def test_tiny_shape_accepted_by_checks(lib):
    assert call_forward(abi.BeamMoeConfig.of(W.TINY), T=0) == abi.BEAM_MOE_OK


def test_shard_range_rejected(lib):
    cfg = cfg_of()
    for lo, hi in ((0, 0), (5, 3), (-1, 4), (0, 257)):
        rc = lib.beam_moe_forward_shard(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, lo, hi, 4, FAKE, None)
        assert rc == abi.BEAM_MOE_ERR_ARG, (lo, hi)
        assert "expert range" in abi.beam_moe_last_error()
    assert lib.beam_moe_forward_shard(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 32, 0, FAKE,
                                      None) == abi.BEAM_MOE_OK


def test_dense_mlp_arguments_checked(lib):
    f = lib.beam_moe_dense_mlp
    assert f(100, 256, FAKE, FAKE, FAKE, FAKE, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(512, 200, FAKE, FAKE, FAKE, FAKE, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(512, 256, FAKE, None, FAKE, FAKE, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(512, 256, FAKE, FAKE, FAKE, FAKE + 8, 4, FAKE, None) == abi.BEAM_MOE_ERR_ALIGN
    assert f(512, 256, FAKE, FAKE, FAKE, FAKE, 0, FAKE, None) == abi.BEAM_MOE_OK


def test_forward_fp8_arguments_checked(lib):
    f = lib.beam_moe_forward_fp8
    cfg = ctypes.byref(cfg_of())
    args = [FAKE] * 9
    assert f(cfg, *args, 0, FAKE, None) == abi.BEAM_MOE_OK
    for i, name in enumerate(["x", "router_w", "expert_bias", "w_gate_q", "gate_scale", "w_up_q", "up_scale",
                              "w_down_q", "down_scale"]):
        bad = list(args)
        bad[i] = None
        assert f(cfg, *bad, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG, name
        assert name in abi.beam_moe_last_error()
        bad[i] = FAKE + 4
        assert f(cfg, *bad, 4, FAKE, None) == abi.BEAM_MOE_ERR_ALIGN, name
    assert f(cfg, *args, 4, None, None) == abi.BEAM_MOE_ERR_ARG


def test_forward_nvfp4_arguments_checked(lib):
    f = lib.beam_moe_forward_nvfp4
    cfg = ctypes.byref(cfg_of())
    args = [FAKE] * 12
    assert f(cfg, *args, 0, FAKE, None) == abi.BEAM_MOE_OK
    for i, name in enumerate(["x", "router_w", "expert_bias", "w_gate_q", "gate_block_scale", "gate_tensor_scale",
                              "w_up_q", "up_block_scale", "up_tensor_scale", "w_down_q", "down_block_scale",
                              "down_tensor_scale"]):
        bad = list(args)
        bad[i] = None
        assert f(cfg, *bad, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG, name
        assert name in abi.beam_moe_last_error()
        bad[i] = FAKE + 4
        assert f(cfg, *bad, 4, FAKE, None) == abi.BEAM_MOE_ERR_ALIGN, name
    assert f(cfg, *args, 4, None, None) == abi.BEAM_MOE_ERR_ARG
    # the 16-element blocks of a 256-wide stage: d and I multiples of 256
    assert f(ctypes.byref(cfg_of(d=384, I=256)), *args, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert "multiples of 256" in abi.beam_moe_last_error()
    assert f(ctypes.byref(cfg_of(d=512, I=384)), *args, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG


def test_forward_host_arguments_checked(lib):
    f = lib.beam_moe_forward_host
    cfg = ctypes.byref(cfg_of())
    w = [FAKE] * 5  # router_w, expert_bias, w_gate, w_up, w_down
    assert f(cfg, None, *w, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG and "x_host" in abi.beam_moe_last_error()
    assert f(cfg, FAKE, *w, 4, None, None) == abi.BEAM_MOE_ERR_ARG and "out_host" in abi.beam_moe_last_error()
    assert f(cfg, FAKE, *w, -1, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(ctypes.byref(cfg_of(top_k=0)), FAKE, *w, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(cfg, FAKE, *w, 0, FAKE, None) == abi.BEAM_MOE_OK


def test_rmsnorm_arguments_checked(lib):
    f = lib.beam_moe_rmsnorm
    eps = ctypes.c_float(1e-6)
    for d in (0, 6, 8192 + 4):
        assert f(d, FAKE, FAKE, eps, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG, d
    assert f(5120, None, FAKE, eps, 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(5120, FAKE, FAKE + 8, eps, 4, FAKE, None) == abi.BEAM_MOE_ERR_ALIGN
    assert f(5120, FAKE, FAKE, ctypes.c_float(float("nan")), 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(5120, FAKE, FAKE, ctypes.c_float(-1.0), 4, FAKE, None) == abi.BEAM_MOE_ERR_ARG
    assert f(5120, FAKE, FAKE, eps, 0, FAKE, None) == abi.BEAM_MOE_OK


def test_sublayer_arguments_checked(lib):
    f = lib.beam_moe_sublayer_forward
    cfg = ctypes.byref(cfg_of())
    eps = ctypes.c_float(1e-6)

    def call(stream_in=FAKE, pre=FAKE, post=FAKE, e=eps, k=5, T=4, out=FAKE, c=cfg):
        return f(c, stream_in, pre, post, e, k, FAKE, FAKE, FAKE, FAKE, FAKE, T, out, None)

    assert call(pre=None) == abi.BEAM_MOE_ERR_ARG and "pre_gamma" in abi.beam_moe_last_error()
    assert call(post=None) == abi.BEAM_MOE_ERR_ARG and "post_gamma" in abi.beam_moe_last_error()
    assert call(stream_in=None) == abi.BEAM_MOE_ERR_ARG and "stream_in" in abi.beam_moe_last_error()
    assert call(out=None) == abi.BEAM_MOE_ERR_ARG and "stream_out" in abi.beam_moe_last_error()
    assert call(k=1) == abi.BEAM_MOE_ERR_ARG and "k=1" in abi.beam_moe_last_error()
    assert call(e=ctypes.c_float(float("inf"))) == abi.BEAM_MOE_ERR_ARG
    assert call(c=ctypes.byref(cfg_of(d=8192 + 128))) == abi.BEAM_MOE_ERR_ARG
    assert call(T=0) == abi.BEAM_MOE_OK


@pytest.mark.parametrize("arg", ["x", "router_w", "expert_bias", "topk_idx", "topk_w"])
def test_route_beam_shape_pointers_checked(lib, arg):
    args = dict(x=FAKE, router_w=FAKE, expert_bias=FAKE, topk_idx=FAKE, topk_w=FAKE)
    args[arg] = None
    assert lib.beam_moe_route(args["x"], args["router_w"], args["expert_bias"], 4, args["topk_idx"],
                              args["topk_w"], None) == abi.BEAM_MOE_ERR_ARG
    assert arg in abi.beam_moe_last_error()
