import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # Build the CUDA library and the oracle in-tree if they are missing or stale
    # (no-ops when up to date).
    from sparse_attention_prefill_tcgen05_gb300 import build as B
    B.build()
    from oracle import oracle as O
    O.build()
