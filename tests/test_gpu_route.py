"""Router parity: the CUDA router against the CPU oracle (indices bit-exact given the GPU's
FP32 logits, near ties reported separately), on Tiny and Beam shapes."""
import json

import numpy as np
import pytest
import torch

import parity as P
from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W

pytestmark = pytest.mark.gpu


def gpu_route(shape, x, wr, b):
    logits = moe.router_logits(x, wr, shape)
    idx, w = moe.route(x, wr, b, shape)
    abi.beam_moe_device_status()
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 7, 128, 129, 300, 1000])
def test_tiny_route_parity(T):
    shape = W.TINY
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda")
    logits, idx, w = gpu_route(shape, x, wr, b)
    P.check_logits(shape, x, wr, logits)
    flagged, _ = P.check_routing(shape, logits, b.cpu().numpy(), idx, w)
    assert len(flagged) <= max(2, T // 100), f"{len(flagged)} near-tie tokens"


@pytest.mark.parametrize("n_group,d,T", [(3, 256, 300), (5, 384, 33), (1, 128, 1000), (8, 512, 4097), (2, 128, 32)])
def test_odd_shape_route_parity(n_group, d, T):
    """Expert counts that are not a multiple of the 128-row weight tile (the tile's last
    rows belong to the next weight piece and must not be stored), short K, ragged token
    tiles, the smallest batch of the tensor-core router (T=33) and the largest of the
    small-batch one (T=32)."""
    shape = W.MoEShape(d=d, I=128, E=32 * n_group, n_group=n_group, topk_group=min(2, n_group), top_k=8)
    x = W.make_tokens(shape, T, 4, "cuda")
    wr, b = W.make_router(shape, 4, "cuda")
    logits, idx, w = gpu_route(shape, x, wr, b)
    P.check_logits(shape, x, wr, logits)
    flagged, _ = P.check_routing(shape, logits, b.cpu().numpy(), idx, w)
    assert len(flagged) <= max(2, T // 100)


@pytest.mark.parametrize("name", ["decode", "prefill", "skewed"])
def test_beam_route_parity(name):
    shape, T, hot = W.WORKLOADS[name]
    x = W.make_tokens(shape, T, 0, "cuda")
    wr, b = W.make_router(shape, 0, "cuda", hot_experts=hot)
    logits, idx, w = gpu_route(shape, x, wr, b)
    sample = W.sample_tokens(T, 512, seed=1).numpy()
    P.check_logits(shape, x[sample], wr, logits[sample])
    flagged, _ = P.check_routing(shape, logits, b.cpu().numpy(), idx, w)
    print(f"{name}: T={T} near-tie tokens {len(flagged)}")
    assert len(flagged) <= max(2, T // 200)
    if hot:
        load = np.bincount(idx.ravel(), minlength=shape.E)
        assert load.max() > 10 * load.mean(), "skewed workload is not skewed"


def test_golden_routing_on_gpu():
    """The hand-worked routing cases, fed through the CUDA router: token j is the one-hot
    vector e_j and router column j holds its logits, so the FP32 logits equal the
    fixture's values exactly."""
    spec = json.load(open(P.__file__.replace("parity.py", "golden/routing_handworked.json")))
    c = spec["config"]
    shape = W.MoEShape(d=128, I=128, E=c["E"], n_group=c["n_group"], topk_group=c["topk_group"], top_k=c["top_k"],
                       scale=c["scale"])
    for case in spec["cases"]:
        bias = torch.full((shape.E,), case["default_bias"], dtype=torch.float32)
        for e, v in case["bias"].items():
            bias[int(e)] = v
        n = len(case["tokens"])
        x = torch.zeros((n, shape.d), dtype=torch.bfloat16)
        wr = torch.zeros((shape.E, shape.d), dtype=torch.float32)
        for j, tok in enumerate(case["tokens"]):
            x[j, j] = 1.0
            wr[:, j] = tok["default_logit"]
            for e, v in tok["logits"].items():
                wr[int(e), j] = v
        logits, idx, w = gpu_route(shape, x.cuda(), wr.cuda(), bias.cuda())
        for j, tok in enumerate(case["tokens"]):
            np.testing.assert_array_equal(logits[j], wr[:, j].numpy())
            assert list(idx[j]) == tok["expect_idx"], (case["name"], idx[j])
            np.testing.assert_allclose(w[j], tok["expect_w"], rtol=2e-6, err_msg=case["name"])


def test_route_deterministic():
    shape, T, _ = W.WORKLOADS["prefill"]
    x = W.make_tokens(shape, T, 3, "cuda")
    wr, b = W.make_router(shape, 3, "cuda")
    a = moe.route(x, wr, b, shape)
    c = moe.route(x, wr, b, shape)
    torch.cuda.synchronize()
    assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_zero_input_routes_to_first_experts():
    shape = W.BEAM
    x = torch.zeros((5, shape.d), dtype=torch.bfloat16, device="cuda")
    wr, _ = W.make_router(shape, 0, "cuda")
    b = torch.full((shape.E,), -0.05, dtype=torch.float32, device="cuda")
    _, idx, w = gpu_route(shape, x, wr, b)
    assert (idx == np.arange(8)[None, :]).all()
    assert (w == np.float32(0.3125)).all()
