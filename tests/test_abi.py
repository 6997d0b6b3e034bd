"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every
symbol include/oop.h declares, and its host-side argument checks reject bad
calls before touching the GPU (no compute call is made here)."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def _declared():
    src = open(os.path.join(ROOT, "include", "oop.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(oop_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def built():
    import ggml_out_prod_gb300 as g
    g.build()
    return g


@needs_nvcc
def test_exports_every_declared_symbol(built):
    L = built.lib()
    names = _declared()
    assert "oop_out_prod" in names and "oop_mul_mat_id_back" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in oop.h but not exported"
    assert set(built.EXPORTS) <= set(names)


@needs_nvcc
def test_status_strings(built):
    for code in range(-12, 1):
        s = built.status_string(code)
        assert s and s != "unknown status"
    assert built.lib().oop_version() >= 1


def _ne(v):
    return (ctypes.c_int64 * len(v))(*v)


@needs_nvcc
@pytest.mark.parametrize("ne_a,ne_b,ne_dst,a_type,want", [
    ((64, 8, 3, 1), (4, 8, 16, 1), (64, 4, 16, 1), 0, -4),     # 16 % 3
    ((64, 8, 1, 2), (4, 8, 1, 3), (64, 4, 1, 3), 0, -4),       # 3 % 2
    ((64, 8, 1, 1), (4, 7, 1, 1), (64, 4, 1, 1), 0, -3),       # K mismatch
    ((64, 8, 1, 1), (4, 8, 1, 1), (64, 5, 1, 1), 0, -3),       # wrong dst ne
    ((48, 8, 1, 1), (4, 8, 1, 1), (48, 4, 1, 1), 8, -3),       # q8_0 M % 32
    ((64, 8, 1, 1), (4, 8, 1, 1), (64, 4, 1, 1), 9, -2),       # q8_1: not a src0 type
    ((64, 8, 1, 1), (4, 8, 1, 1), (64, 4, 1, 1), 99, -2),      # unknown type
    ((128, 8, 1, 1), (4, 8, 1, 1), (128, 4, 1, 1), 12, -3),    # q4_K M % 256
    ((64, -1, 1, 1), (4, -1, 1, 1), (64, 4, 1, 1), 0, -3),     # negative size
    ((64, 8, 0, 1), (4, 8, 0, 1), (64, 4, 0, 1), 0, -4),       # ne02 = 0
])
def test_host_checks(built, ne_a, ne_b, ne_dst, a_type, want):
    L = built.lib()
    dummy = ctypes.c_void_p(0x1000)
    rc = L.oop_out_prod(dummy, a_type, dummy, dummy, _ne(ne_a), _ne(ne_b), _ne(ne_dst),
                        None, 0, None)
    assert rc == want


@needs_nvcc
def test_host_checks_nulls(built):
    L = built.lib()
    rc = L.oop_out_prod(None, 0, None, None, _ne((64, 8, 1, 1)), _ne((4, 8, 1, 1)),
                        _ne((64, 4, 1, 1)), None, 0, None)
    assert rc == -1
    rc = L.oop_out_prod(None, 0, None, None, None, _ne((4, 8, 1, 1)), _ne((64, 4, 1, 1)),
                        None, 0, None)
    assert rc == -1
    # misaligned dst
    rc = L.oop_out_prod(ctypes.c_void_p(0x1000), 0, ctypes.c_void_p(0x1000),
                        ctypes.c_void_p(0x1002), _ne((64, 8, 1, 1)), _ne((4, 8, 1, 1)),
                        _ne((64, 4, 1, 1)), None, 0, None)
    assert rc == -5
    # empty dst: nothing to do, no device needed
    rc = L.oop_out_prod(None, 0, None, None, _ne((64, 8, 1, 1)), _ne((0, 8, 1, 1)),
                        _ne((64, 0, 1, 1)), None, 0, None)
    assert rc == 0
    # MUL_MAT_ID_BACK: wrong type (q8_1 is no expert type), blocks that do not
    # fill K, negative size
    rc = L.oop_mul_mat_id_back(None, 9, None, None, None, _ne((4, 3, 2)), _ne((1, 1)),
                               None, 0, None)
    assert rc == -2
    rc = L.oop_mul_mat_id_back(None, 8, None, None, None, _ne((48, 3, 2)), _ne((1, 1)),
                               None, 0, None)
    assert rc == -3
    rc = L.oop_mul_mat_id_back(None, 0, None, None, None, _ne((4, -3, 2)), _ne((1, 1)),
                               None, 0, None)
    assert rc == -3


def test_oracle_is_not_linked_by_product():
    """The product package never imports, loads or links the oracle."""
    pkg = os.path.join(ROOT, "ggml_out_prod_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                for bad in ("import oracle", "from oracle", "liboracle", "oracle.h"):
                    assert bad not in txt, f"{f} refers to the oracle ({bad})"
