import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def beam_experts():
    """Beam-shaped expert weights (seed 0) on cuda:0, shared by every GPU test (20 GB)."""
    from sparse_moe_transformer_bias_b300 import workloads as W
    return W.make_experts(W.BEAM, seed=0, device="cuda")


@pytest.fixture(scope="session")
def beam_host_cache():
    """Host copies (BF16 bits) of Beam experts handed to the oracle, filled on demand."""
    return {}
