import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on CPU")


def pytest_sessionstart(session):
    # The product tests load the in-tree library; (re)build it when sources changed.  nvcc
    # cross-compiles for sm_103a without a GPU, so this also works on CPU-only hosts.
    import importlib.util
    path = os.path.join(ROOT, "prefix_shared_kv_token_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_pkv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
