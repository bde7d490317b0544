import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def _ensure_library_built():
    import importlib.util
    path = os.path.join(ROOT, "lm_head_loss_gb300", "build_lib.py")
    spec = importlib.util.spec_from_file_location("_flce_build_lib_conftest", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


_ensure_library_built()
