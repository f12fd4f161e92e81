"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import pins
from oracle import oracle as O


@pytest.fixture(scope="module")
def orc():
    return O.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_rejects_bad_config(orc):
    from sparse_moe_transformer_bias_b300 import workloads as W
    assert orc.check_cfg(W.BEAM) and orc.check_cfg(W.TINY)
    assert not orc.check_cfg(W.MoEShape(E=250))                 # E not a multiple of n_group
    assert not orc.check_cfg(W.MoEShape(topk_group=9))          # more kept groups than groups
    assert not orc.check_cfg(W.MoEShape(n_group=8, topk_group=1, top_k=33))  # more picks than candidates
