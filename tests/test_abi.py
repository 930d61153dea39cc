"""The C-ABI libraries load on a CPU-only machine and export every symbol their
headers declare (no compute calls here)."""
import ctypes
import pathlib
import re

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _declared(header: pathlib.Path):
    text = header.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fi_[a-z0-9_]+)\s*\(", text)))


@pytest.mark.parametrize("header,libname", [
    ("fi_nvfp4.h", "libfi_nvfp4.so"),
    ("fi_nvfp4_diag.h", "libfi_nvfp4_diag.so"),
])
def test_library_exports_every_declared_symbol(header, libname):
    names = _declared(ROOT / "include" / header)
    assert names, header
    lib = ctypes.CDLL(str(ROOT / "nvfp4_paged_kv_slot_b300" / libname))
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_match_headers():
    import nvfp4_paged_kv_slot_b300 as fi
    import nvfp4_paged_kv_slot_b300.diag as diag
    assert sorted(fi.EXPORTED) == _declared(ROOT / "include" / "fi_nvfp4.h")
    assert sorted(diag.EXPORTED) == _declared(ROOT / "include" / "fi_nvfp4_diag.h")


def test_host_only_calls_work_without_gpu():
    import nvfp4_paged_kv_slot_b300 as fi
    assert fi.fi_version() >= 100
    assert fi.lib.fi_status_string(fi.FI_ERR_BAD_SCALE).decode().startswith("global decode")
    info, work = fi.fi_prefill_plan_host([0, 3], [0, 3], 4, 2, 64, 16)
    assert info["num_units"] == work.shape[0] == 2   # one unit per kv head (G = 2)


def test_oracle_is_not_imported_by_the_product():
    """The product package and its sources never reference the oracle."""
    pkg = ROOT / "nvfp4_paged_kv_slot_b300"
    for p in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + \
            list(pkg.rglob("*.cpp")) + list(pkg.rglob("*.h")):
        text = p.read_text()
        assert "import oracle" not in text and "from oracle" not in text, p
        assert "oracle.h" not in text and "liboracle" not in text, p
