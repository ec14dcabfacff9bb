"""Shared pytest configuration: markers, import paths, and the library build."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def attn_lib():
    """The C library, built in-tree with nvcc first if it is missing or stale."""
    from transformer_scaled_dot_fwd_gb300 import build as _build
    import transformer_scaled_dot_fwd_gb300 as attn
    _build.build(quiet=True)
    return attn.lib()


@pytest.fixture(scope="session")
def gpu(attn_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
