import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); run with -m gpu")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


def build_library():
    """Compile libxsattn.so if stale (by path, without importing the package)."""
    import importlib.util
    path = os.path.join(ROOT, "dit_attention_ulysses_gb300", "_build.py")
    spec = importlib.util.spec_from_file_location("xsattn_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
