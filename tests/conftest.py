import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _load_build_script():
    """The package's build script, loaded by path (importing the package itself
    needs the library that this script builds)."""
    path = os.path.join(ROOT, "nvfp4_paged_kv_slot_b300", "build.py")
    spec = importlib.util.spec_from_file_location("_fi_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
    # Compile the C-ABI libraries (sm_103a, cross-compiled without a GPU) and
    # the CPU oracle if their sources changed.
    _load_build_script().build()
    from oracle import build as oracle_build
    oracle_build.build()


@pytest.fixture(scope="session")
def oracle():
    import oracle as O
    O.lib()
    return O
