import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def build_library():
    """Compile the CUDA library in-tree (no-op when up to date)."""
    import __graft_entry__
    __graft_entry__.build()


def build_checked_library() -> str:
    """Compile the bounds-checked variant of the library (liblatent_moe_checked.so)."""
    import importlib.util
    path = os.path.join(ROOT, "latent_mixture_experts_router_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_lmoe_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(checked=True)
