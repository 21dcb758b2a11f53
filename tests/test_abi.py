"""The C ABI library builds for sm_103a, loads, and exports every entry point
declared in include/smp.h (no GPU needed; no compute call is made)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "smp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(smp_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from top_selection_stats_gb300 import build, binding
    build.build()
    return binding.load_library()


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("smp_create", "smp_destroy", "smp_topk_topp_mask", "smp_sample", "smp_argmax"):
        assert n in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.smp_status_string(0) == b"ok"
    assert b"empty" in lib.smp_status_string(1)
    assert lib.smp_status_string(99) == b"unknown status"


def test_null_handle_is_rejected_without_device_work(lib):
    # argument checks happen before any CUDA call
    assert lib.smp_set_row_info(None, None) == 3
    assert lib.smp_destroy(None) == 0
    assert lib.smp_create(None, 0, 1, 1) == 3
    assert lib.smp_spec_verify(None, None, None, None, 1, 1, 8, 8, None, None, None, None, None,
                               None) == 3


def test_binding_fails_loudly_without_library(tmp_path):
    from top_selection_stats_gb300 import binding
    with pytest.raises(FileNotFoundError):
        binding.load_library(str(tmp_path / "missing.so"))
