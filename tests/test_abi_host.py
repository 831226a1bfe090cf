"""Host-side checks that need no GPU: the C ABI loads and exports every
function include/bigemm.h declares; argument validation rejects bad calls
before any device work; the product path has no CPU fallback."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bigemm.h")


@pytest.fixture(scope="module")
def lib():
    sys.path.insert(0, ROOT)
    from broadcast_implicit_gemm_gb300 import _build
    _build.build()
    import broadcast_implicit_gemm_gb300 as bg
    return bg.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z][a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("conv2d_nchw_plan", "conv2d_nchw_run", "bcast_nchw_run", "conv2d_nchw_plan_destroy",
              "bigemm_status_string", "bigemm_last_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    import broadcast_implicit_gemm_gb300 as bg
    assert bg.bigemm_status_string(0) == "ok"
    assert "invalid" in bg.bigemm_status_string(1)
    assert "timed out" in bg.bigemm_status_string(4)
    assert bg.bigemm_version().startswith("bigemm")


@pytest.mark.parametrize("args", [
    (1, 2, 2, 8, 8, 3, 3, 1, 0, 1),     # window larger than the padded input: Ho <= 0
    (0, 8, 8, 8, 8, 3, 3, 1, 1, 1),     # N = 0
    (1, 8, 8, 8, 8, 3, 3, 0, 1, 1),     # stride 0
    (1, 8, 8, 8, 8, 3, 3, 1, -1, 1),    # negative padding
    (1, 8, 8, 9, 8, 3, 3, 1, 1, 2),     # CO not divisible by groups
    (1, 8, 8, 8, 6, 3, 3, 1, 1, 4),     # CI not divisible by groups
])
def test_plan_rejects_invalid_shapes_without_a_device(lib, args):
    h = ctypes.c_void_p()
    st = lib.conv2d_nchw_plan(*args, 0, 0, 0, 0, None, ctypes.byref(h))
    assert st == 1 and not h.value


def test_plan_rejects_bad_dtype_and_epilogue(lib):
    h = ctypes.c_void_p()
    assert lib.conv2d_nchw_plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 7, 0, 0, 0, None, ctypes.byref(h)) == 1
    assert lib.conv2d_nchw_plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 0, 0, 9, 0, None, ctypes.byref(h)) == 1
    assert lib.conv2d_nchw_plan(1, 8, 8, 8, 8, 3, 3, 1, 1, 1, 0, 0, 0, 0, None, None) == 1


def test_bcast_rejects_bad_arguments(lib):
    assert lib.bcast_nchw_run(0, 4, 4, 4, 1, 16, 1e-5, 16, 0, None) == 1
    assert lib.bcast_nchw_run(1, 4, 4, 4, 9, 16, 1e-5, 16, 0, None) == 1
    assert lib.bcast_nchw_run(1, 4, 4, 4, 1, None, 1e-5, 16, 0, None) == 1
    assert lib.bcast_nchw_run(1, 4, 4, 4, 1, 16, 1e-5, 16, 5, None) == 1
    assert lib.conv2d_nchw_run(None, 16, 16, None, 0.0, 16, None) == 1
    assert lib.conv2d_nchw_plan_destroy(None) == 1


def test_missing_library_fails_loudly():
    code = ("import os, sys; sys.path.insert(0, %r); os.environ['BIGEMM_LIB']='/nonexistent/lib.so';"
            "import broadcast_implicit_gemm_gb300 as bg\n"
            "try:\n  bg.bcast_nchw_run(1,1,1,1,1,0,0.0,0,0,0)\nexcept RuntimeError as e:\n"
            "  print('raised', e)\n") % ROOT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert "raised" in r.stdout and "missing" in r.stdout


def test_product_path_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "broadcast_implicit_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|liboracle|oracle\.c)", text), f


def _c_struct_fields(name):
    """Field names of a typedef'd C struct in the header, in order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"typedef\s+struct\s*\{(.*?)\}\s*" + name + r"\s*;", text, flags=re.S)
    assert m, name
    return re.findall(r"\b([a-z_][a-z0-9_]*)\s*;", m.group(1))


def test_plan_options_binding_matches_header():
    # the ctypes mirror must list the header's int fields in the same order
    sys.path.insert(0, ROOT)
    import broadcast_implicit_gemm_gb300 as bg
    assert [f for f, _ in bg.PlanOptions._fields_] == _c_struct_fields("bigemm_plan_options")
    assert all(t is ctypes.c_int for _, t in bg.PlanOptions._fields_)


def test_enum_values_match_header():
    # the binding's epilogue, broadcast-op and mode constants equal the header's
    sys.path.insert(0, ROOT)
    import broadcast_implicit_gemm_gb300 as bg
    text = open(HEADER).read()
    vals = dict((k, int(v)) for k, v in re.findall(r"\b(BIGEMM_[A-Z0-9_]+)\s*=\s*(\d+)", text))
    for name in ("EPI_NONE", "EPI_BIAS", "EPI_BIAS_EXP", "EPI_BIAS_RSQRT", "EPI_BIAS_RECIP", "EPI_BIAS_RELU",
                 "BC_COPY", "BC_EXP", "BC_RSQRT", "BC_RECIP", "KIND_UMMA", "KIND_SIMT"):
        assert getattr(bg, name) == vals["BIGEMM_" + name], name
