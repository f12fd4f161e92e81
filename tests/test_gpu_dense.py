"""Dense SwiGLU MLP of the first decoder layers through the C ABI against the CPU oracle's
expert (the same SwiGLU written out in FP64). The pages give no width for these layers, so
the widths here are test choices."""
import numpy as np
import pytest
import torch

import parity as P
from oracle import oracle as O
from sparse_moe_transformer_bias_b300 import abi, moe

pytestmark = pytest.mark.gpu


def dense_inputs(d, I, T, seed):
    g = torch.Generator(device="cuda").manual_seed(500 + seed)
    x = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    wg = (torch.randn((I, d), generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    wu = (torch.randn((I, d), generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    wd = (torch.randn((d, I), generator=g, device="cuda") / I ** 0.5).to(torch.bfloat16)
    return x, wg, wu, wd


@pytest.mark.parametrize("d,I,T,n_check", [(512, 1024, 1, 1), (512, 1024, 33, 33), (512, 256, 300, 300),
                                           (5120, 10240, 16, 16), (5120, 10240, 1000, 12)])
def test_dense_mlp_parity(d, I, T, n_check):
    x, wg, wu, wd = dense_inputs(d, I, T, seed=d + I + T)
    out = moe.dense_mlp(x, wg, wu, wd)
    abi.beam_moe_device_status()
    tokens = np.unique(np.linspace(0, T - 1, n_check).astype(int))
    shape = type("S", (), {"d": d, "I": I})
    xb, gb, ub, db = (O.bf16_bits(t) for t in (x, wg, wu, wd))
    ref = np.stack([O.expert(shape, (xb[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64), gb, ub, db)
                    for t in tokens])
    frob = P.check_output(out.float().cpu().numpy()[tokens], ref, f"dense d={d} I={I} T={T}")
    print(f"dense d={d} I={I} T={T}: rel frob {frob:.2e}")


def test_dense_mlp_deterministic_and_launches():
    x, wg, wu, wd = dense_inputs(512, 512, 257, seed=1)
    a = moe.dense_mlp(x, wg, wu, wd)
    b = moe.dense_mlp(x, wg, wu, wd)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert abi.beam_moe_last_launch_count() == 2
