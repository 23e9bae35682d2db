import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the CUDA library")


def read_golden(name):
    """key value pairs of a tests/golden fixture (comments start with #)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split(None, 1)
                out[k] = v.strip()
    return out


# ------------------------------------------------------------ GPU fixtures --

ARENA_SEED = 0
ARENA_SCALE_LO, ARENA_SCALE_HI = 118, 128


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def arena(cuda_dev):
    """All 896 routed experts of the seeded workload, back to back in one
    device buffer (about 15.7 GB), and their pointer table."""
    import synth
    import mxfp4_routed_expert_k3mx_gb300 as k3mx
    buf = synth.expert_arena_device(cuda_dev, seed=ARENA_SEED, lo=ARENA_SCALE_LO, hi=ARENA_SCALE_HI)
    table = k3mx.expert_table(buf)
    return buf, table
