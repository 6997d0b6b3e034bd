"""CPU oracle for OUT_PROD and MUL_MAT_ID_BACK (plain C, fp64 accumulation).

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports, links or runs anything here, and nothing here imports the product.

``build()`` compiles ``oracle.c`` with gcc (OpenMP) into ``oracle/_build``.
The wrappers take numpy arrays in ggml layout: a tensor with
ne = {ne0, ne1, ne2, ne3} is an array of shape (ne3, ne2, ne1, ne0); quantised
src0 is a uint8 array whose last axis holds the row bytes.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(exact integer brute force, the rank-one closed form, linearity, broadcast as
explicit replication, numpy's own binary16 decoder, quantiser round trips,
one-hot routing against the dense backward, and finite differences of the
forward product).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")

_lock = threading.Lock()
_lib = None

F32, F16, Q4_0, Q8_0, BF16 = 0, 1, 2, 8, 30

_i64p = ctypes.POINTER(ctypes.c_int64)
_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2 -fopenmp); returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_half_to_double.restype = ctypes.c_double
            L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_round_to_half.restype = ctypes.c_double
            L.oracle_round_to_half.argtypes = [ctypes.c_double]
            L.oracle_dequant_row.argtypes = [ctypes.c_int, _vp, ctypes.c_int64, _dp]
            L.oracle_out_prod.argtypes = [_vp, ctypes.c_int, _fp, _i64p, _i64p,
                                          _fp, _dp, _dp, ctypes.c_int]
            L.oracle_out_prod_at.argtypes = [_vp, ctypes.c_int, _fp, _i64p, _i64p,
                                             _i64p, ctypes.c_int64, _dp, _dp,
                                             ctypes.c_int]
            L.oracle_out_prod_fp16_staged.argtypes = [_vp, ctypes.c_int, _fp, _i64p,
                                                      _i64p, _fp, ctypes.c_int]
            L.oracle_mul_mat_id_back.argtypes = [_vp, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int32), _fp,
                                                 _i64p, _i64p, _fp, _dp, _dp,
                                                 ctypes.c_int]
            L.oracle_mul_mat_id_back_at.argtypes = [_vp, ctypes.c_int,
                                                    ctypes.POINTER(ctypes.c_int32),
                                                    _fp, _i64p, _i64p, _i64p,
                                                    ctypes.c_int64, _dp, _dp,
                                                    ctypes.c_int]
            L.oracle_mul_mat.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, _dp]
            L.oracle_out_prod_strided.argtypes = [_vp, ctypes.c_int, _vp, _i64p, _i64p,
                                                  _i64p, _fp, _dp, _dp, ctypes.c_int]
            L.oracle_mul_mat_back.argtypes = [_vp, ctypes.c_int, _fp, _fp, _i64p, _i64p,
                                              _fp, _dp, _dp, _fp, _dp, _dp, ctypes.c_int]
            L.oracle_mul_mat_id_weight_grad.argtypes = [_fp, ctypes.POINTER(ctypes.c_int32), _fp,
                                                        _i64p, _i64p, ctypes.c_int64, _fp, _dp,
                                                        _dp, ctypes.c_int]
            _lib = L
    return _lib


def _ne(v):
    return (ctypes.c_int64 * len(v))(*[int(x) for x in v])


def _ptr(x, ctype):
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def _vptr(x):
    return ctypes.c_void_p(x.ctypes.data) if x is not None and x.size else None


def ne_of(arr: np.ndarray, type_id: int = F32, ne0: int | None = None):
    """ggml ne of an array in this layout (quantised rows need ``ne0``)."""
    shp = (1,) * (4 - arr.ndim) + tuple(arr.shape)
    if type_id in (Q8_0, Q4_0):
        assert ne0 is not None
        return (ne0, shp[2], shp[1], shp[0])
    return (shp[3], shp[2], shp[1], shp[0])


def half_to_double(h: int) -> float:
    return lib().oracle_half_to_double(int(h))


def bf16_to_double(h: int) -> float:
    return lib().oracle_bf16_to_double(int(h))


def round_to_half(x: float) -> float:
    return lib().oracle_round_to_half(float(x))


def dequant_row(type_id: int, row: np.ndarray, n: int) -> np.ndarray:
    row = np.ascontiguousarray(row)
    out = np.empty(n, dtype=np.float64)
    rc = lib().oracle_dequant_row(type_id, _vptr(row), n, _ptr(out, ctypes.c_double))
    if rc:
        raise ValueError("oracle_dequant_row rejected its arguments")
    return out


def out_prod(a, a_type, b, ne_a, ne_b, nthreads=0, want=("dst", "f64", "abs")):
    """Whole-tensor OUT_PROD.  Returns a dict with the requested outputs, each
    shaped (ne13, ne12, N, M)."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b, dtype=np.float32)
    M, N, n2, n3 = ne_a[0], ne_b[0], ne_b[2], ne_b[3]
    shape = (n3, n2, N, M)
    dst = np.empty(shape, np.float32) if "dst" in want else None
    f64 = np.empty(shape, np.float64) if "f64" in want else None
    ab = np.empty(shape, np.float64) if "abs" in want else None
    rc = lib().oracle_out_prod(
        _vptr(a), a_type, _ptr(b, ctypes.c_float) if b.size else None, _ne(ne_a),
        _ne(ne_b), _ptr(dst, ctypes.c_float) if dst is not None else None,
        _ptr(f64, ctypes.c_double) if f64 is not None else None,
        _ptr(ab, ctypes.c_double) if ab is not None else None, nthreads)
    if rc:
        raise ValueError("oracle_out_prod rejected its arguments")
    return {"dst": dst, "f64": f64, "abs": ab}


def out_prod_fp16_staged(a, a_type, b, ne_a, ne_b, nthreads=0):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b, dtype=np.float32)
    M, N, n2, n3 = ne_a[0], ne_b[0], ne_b[2], ne_b[3]
    dst = np.empty((n3, n2, N, M), np.float32)
    rc = lib().oracle_out_prod_fp16_staged(
        _vptr(a), a_type, _ptr(b, ctypes.c_float), _ne(ne_a), _ne(ne_b),
        _ptr(dst, ctypes.c_float), nthreads)
    if rc:
        raise ValueError("oracle_out_prod_fp16_staged rejected its arguments")
    return dst


def out_prod_at(a, a_type, b, ne_a, ne_b, coords, nthreads=0):
    """OUT_PROD at (m, n, i2, i3) rows of ``coords``: (value_f64, abssum)."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b, dtype=np.float32)
    coords = np.ascontiguousarray(coords, dtype=np.int64).reshape(-1, 4)
    val = np.empty(len(coords), np.float64)
    ab = np.empty(len(coords), np.float64)
    rc = lib().oracle_out_prod_at(
        _vptr(a), a_type, _ptr(b, ctypes.c_float), _ne(ne_a), _ne(ne_b),
        _ptr(coords, ctypes.c_int64), len(coords), _ptr(val, ctypes.c_double),
        _ptr(ab, ctypes.c_double), nthreads)
    if rc:
        raise ValueError("oracle_out_prod_at rejected its arguments")
    return val, ab


def mul_mat_id_back(W, w_type, ids, g, ne_w, nthreads=0):
    """dx (float32, fp64 sum, abssum), each shaped (n_tokens, n_used, K).
    ``ids`` is int32 [n_tokens, n_used]."""
    W = np.ascontiguousarray(W)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    n_tok, n_used = ids.shape
    K = ne_w[0]
    dx = np.empty((n_tok, n_used, K), np.float32)
    f64 = np.empty((n_tok, n_used, K), np.float64)
    ab = np.empty((n_tok, n_used, K), np.float64)
    rc = lib().oracle_mul_mat_id_back(
        _vptr(W), w_type, _ptr(ids, ctypes.c_int32), _ptr(g, ctypes.c_float),
        _ne(ne_w), _ne((n_used, n_tok)), _ptr(dx, ctypes.c_float),
        _ptr(f64, ctypes.c_double), _ptr(ab, ctypes.c_double), nthreads)
    if rc:
        raise ValueError("oracle_mul_mat_id_back rejected its arguments")
    return {"dst": dx, "f64": f64, "abs": ab}


def mul_mat_id_back_at(W, w_type, ids, g, ne_w, coords, nthreads=0):
    """MUL_MAT_ID_BACK at (k, i, t) rows of ``coords``: (value_f64, abssum)."""
    W = np.ascontiguousarray(W)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    n_tok, n_used = ids.shape
    coords = np.ascontiguousarray(coords, dtype=np.int64).reshape(-1, 3)
    val = np.empty(len(coords), np.float64)
    ab = np.empty(len(coords), np.float64)
    rc = lib().oracle_mul_mat_id_back_at(
        _vptr(W), w_type, _ptr(ids, ctypes.c_int32), _ptr(g, ctypes.c_float),
        _ne(ne_w), _ne((n_used, n_tok)), _ptr(coords, ctypes.c_int64), len(coords),
        _ptr(val, ctypes.c_double), _ptr(ab, ctypes.c_double), nthreads)
    if rc:
        raise ValueError("oracle_mul_mat_id_back_at rejected its arguments")
    return val, ab


def mul_mat(W, x):
    """Forward product in fp64: W (R, K) rows = ggml {K, R}; x (T, K);
    returns y (T, R) with y[t, r] = sum_k W[r, k] x[t, k]."""
    W = np.ascontiguousarray(W, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    R, K = W.shape
    T = x.shape[0]
    y = np.empty((T, R), np.float64)
    rc = lib().oracle_mul_mat(_ptr(W, ctypes.c_double), _ptr(x, ctypes.c_double),
                              K, R, T, _ptr(y, ctypes.c_double))
    if rc:
        raise ValueError("oracle_mul_mat rejected its arguments")
    return y


def view_ne_nb(b):
    """ggml ne and byte strides nb of a float32 numpy view with shape
    (ne3, ne2, ne1, ne0) (fewer axes allowed); strides must be >= 0."""
    b = np.asarray(b)
    shp = (1,) * (4 - b.ndim) + tuple(b.shape)
    st = (0,) * (4 - b.ndim) + tuple(b.strides)
    ne = (shp[3], shp[2], shp[1], shp[0])
    nb = (st[3], st[2], st[1], st[0])
    if any(x < 0 for x in nb):
        raise ValueError("negative strides are not supported")
    return ne, nb


def out_prod_strided(a, a_type, b_view, ne_a, nthreads=0):
    """OUT_PROD with src1 read through the strides of the float32 numpy view
    ``b_view`` (shape (ne13, ne12, K, N), any non-negative strides).  Returns
    the same dict as out_prod."""
    a = np.ascontiguousarray(a)
    if b_view.dtype != np.float32:
        raise ValueError("b must be float32")
    ne_b, nb_b = view_ne_nb(b_view)
    M, N, n2, n3 = ne_a[0], ne_b[0], ne_b[2], ne_b[3]
    shape = (n3, n2, N, M)
    dst = np.empty(shape, np.float32)
    f64 = np.empty(shape, np.float64)
    ab = np.empty(shape, np.float64)
    bp = ctypes.c_void_p(b_view.ctypes.data) if b_view.size else None
    rc = lib().oracle_out_prod_strided(
        _vptr(a), a_type, bp, _ne(nb_b), _ne(ne_a), _ne(ne_b),
        _ptr(dst, ctypes.c_float), _ptr(f64, ctypes.c_double), _ptr(ab, ctypes.c_double),
        nthreads)
    if rc:
        raise ValueError("oracle_out_prod_strided rejected its arguments")
    return {"dst": dst, "f64": f64, "abs": ab}


def mul_mat_back(W, w_type, x, dy, ne_w, nthreads=0):
    """Both gradients of y = MUL_MAT(W, x) given dy.  W: src0 bytes or array of
    ggml shape ne_w = {K, R, ne02, ne03}; x: float32 (ne13, ne12, T, K);
    dy: float32 (ne13, ne12, T, R).  Returns {"dx": {...}, "dW": {...}}, each
    with "dst", "f64" and "abs" (dx shaped like x, dW (ne03, ne02, R, K))."""
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x, dtype=np.float32)
    dy = np.ascontiguousarray(dy, dtype=np.float32)
    ne_x = ne_of(x)
    K, R, n02, n03 = ne_w
    out = {}
    for name, shape in (("dx", (ne_x[3], ne_x[2], ne_x[1], K)), ("dW", (n03, n02, R, K))):
        out[name] = {"dst": np.empty(shape, np.float32), "f64": np.empty(shape, np.float64),
                     "abs": np.empty(shape, np.float64)}
    rc = lib().oracle_mul_mat_back(
        _vptr(W), w_type, _ptr(x, ctypes.c_float), _ptr(dy, ctypes.c_float), _ne(ne_w),
        _ne(ne_x), _ptr(out["dW"]["dst"], ctypes.c_float),
        _ptr(out["dW"]["f64"], ctypes.c_double), _ptr(out["dW"]["abs"], ctypes.c_double),
        _ptr(out["dx"]["dst"], ctypes.c_float), _ptr(out["dx"]["f64"], ctypes.c_double),
        _ptr(out["dx"]["abs"], ctypes.c_double), nthreads)
    if rc:
        raise ValueError("oracle_mul_mat_back rejected its arguments")
    return out


def mul_mat_id_weight_grad(x, ids, dy, E, nthreads=0):
    """Expert-weight gradient of MUL_MAT_ID.  x: float32 (n_tokens, n_x, K);
    ids: int32 (n_tokens, n_used); dy: float32 (n_tokens, n_used, N).
    Returns {"dst", "f64", "abs"}, each shaped (E, N, K) (ggml {K, N, E})."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    dy = np.ascontiguousarray(dy, dtype=np.float32)
    T, n_x, K = x.shape
    _, n_used, N = dy.shape
    shape = (E, N, K)
    out = {"dst": np.empty(shape, np.float32), "f64": np.empty(shape, np.float64),
           "abs": np.empty(shape, np.float64)}
    rc = lib().oracle_mul_mat_id_weight_grad(
        _ptr(x, ctypes.c_float), _ptr(ids, ctypes.c_int32), _ptr(dy, ctypes.c_float),
        _ne((K, n_x, T)), _ne((N, n_used, T)), int(E), _ptr(out["dst"], ctypes.c_float),
        _ptr(out["f64"], ctypes.c_double), _ptr(out["abs"], ctypes.c_double), nthreads)
    if rc:
        raise ValueError("oracle_mul_mat_id_weight_grad rejected its arguments")
    return out
