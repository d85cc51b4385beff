"""The C-ABI library builds, loads without a GPU and exports every entry
point that include/*.h declares (no compute calls: CPU only)."""
import ctypes
import glob
import os
import re

import pytest

from paged_mla_speculative_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_verify_\w+)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["mla_verify_plan_create", "mla_verify_attn", "mla_verify_attn_host",
              "mla_verify_plan_destroy", "mla_verify_get_error", "mla_verify_strerror"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert declared_functions() == set(binding.SIGNATURES)


def test_version_and_strerror_without_gpu():
    lib = binding.load_library()
    assert lib.mla_verify_version() >= 100
    assert binding.strerror(0) == "ok"
    assert "aligned" in binding.strerror(-2)
    assert binding.strerror(12345) == "unknown status"


def test_plan_create_rejects_bad_shapes_before_touching_a_gpu():
    lib = binding.load_library()
    h = ctypes.c_void_p()
    # T = 0, T = 33, page size 16, out dtype 7: rejected on the host.
    assert lib.mla_verify_plan_create(ctypes.byref(h), 1, 0, 16, 1, 1024, 300, 0, 0) == -3
    assert lib.mla_verify_plan_create(ctypes.byref(h), 1, 33, 16, 1, 1024, 300, 0, 0) == -3
    assert lib.mla_verify_plan_create(ctypes.byref(h), 1, 4, 16, 16, 1024, 300, 0, 0) == -3
    assert lib.mla_verify_plan_create(ctypes.byref(h), 1, 4, 16, 1, 1024, 300, 7, 0) == -3
    assert lib.mla_verify_plan_create(None, 1, 4, 16, 1, 1024, 300, 0, 0) == -1


def test_null_plan_is_rejected():
    lib = binding.load_library()
    assert lib.mla_verify_attn(None, 1, None, None, None, None, None, None,
                               ctypes.c_float(0.1), None, None, None) == -1
    assert lib.mla_verify_plan_get_nsplit(None, 1) == -1
    w, st = ctypes.c_int(), ctypes.c_int()
    assert lib.mla_verify_plan_get_pack_schedule(None, 1, ctypes.byref(w), ctypes.byref(st)) == -1
    assert lib.mla_verify_plan_inject_fault(None, 1) == -1
    lib.mla_verify_plan_destroy(None)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_mla_speculative_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        src = open(f).read()
        assert "import oracle" not in src and "from oracle" not in src, f
