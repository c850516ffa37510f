import json
import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name: str) -> dict:
    with open(GOLDEN / name) as f:
        return json.load(f)


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if it is missing (nvcc cross-compiles here)."""
    from dsa_sparse_attention_fp8_gb300 import _build
    _build.build_library(quiet=True)
    from dsa_sparse_attention_fp8_gb300 import binding
    return binding.load()
