"""GB300 OUT_PROD and MUL_MAT_ID_BACK: a thin Python binding of ``liboop.so``.

The binding only marshals arguments: torch tensors give device pointers, ggml
``ne`` and the current stream; every step of the computation runs in the CUDA
library.  There is no fallback: if the library is not built, or the device is
not an sm_103 GPU, calls raise.

Layout: a ggml tensor with ne = {ne0, ne1, ne2, ne3} is a contiguous torch
tensor of shape (ne3, ne2, ne1, ne0) (trailing dims may be dropped); a
quantised src0 is a uint8 tensor whose last axis holds one row's bytes.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

TYPE_F32 = 0
TYPE_F16 = 1
TYPE_Q4_0 = 2
TYPE_Q4_1 = 3
TYPE_Q5_0 = 6
TYPE_Q5_1 = 7
TYPE_Q8_0 = 8
TYPE_Q2_K = 10
TYPE_Q3_K = 11
TYPE_Q4_K = 12
TYPE_Q5_K = 13
TYPE_Q6_K = 14
TYPE_BF16 = 30

PATH_AUTO = 0
PATH_SKINNY = 1
PATH_TCGEN05 = 2
PATH_SIMT = 3

HAS_TCGEN05 = True

# schedules of the tensor-core tile kernel (set_tc_schedule, a test hook)
SCHEDULE_AUTO = 0
SCHEDULE_DATA_PARALLEL = 1
SCHEDULE_STREAM_K = 2

OK = 0
ERR_NULL = -1
ERR_TYPE = -2
ERR_SHAPE = -3
ERR_BROADCAST = -4
ERR_ALIGN = -5
ERR_WORKSPACE = -6
ERR_CUDA = -7
ERR_BAD_ID = -8
ERR_DEVICE_TIMEOUT = -9
ERR_DEVICE = -10
ERR_PATH = -11
ERR_SCRATCH_LIMIT = -12

# (elements, bytes) per block of the quantised types; the plain 16-bit types
# are tensors of 2-byte elements
_BLOCKS = {TYPE_Q4_0: (32, 18), TYPE_Q4_1: (32, 20), TYPE_Q5_0: (32, 22),
           TYPE_Q5_1: (32, 24), TYPE_Q8_0: (32, 34), TYPE_Q2_K: (256, 84),
           TYPE_Q3_K: (256, 110), TYPE_Q4_K: (256, 144), TYPE_Q5_K: (256, 176),
           TYPE_Q6_K: (256, 210)}
_HALF_TYPES = (TYPE_F16, TYPE_BF16)

_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p

EXPORTS = (
    "oop_out_prod", "oop_out_prod_ex", "oop_out_prod_workspace_size",
    "oop_mul_mat_id_back", "oop_mul_mat_id_back_ex", "oop_mul_mat_id_back_workspace_size",
    "oop_device_status", "oop_status_string", "oop_version", "oop_debug_inject_timeout",
    "oop_last_cuda_error", "oop_out_prod_noalloc", "oop_out_prod_noalloc_scratch_bytes",
    "oop_profile_main_kernel", "oop_out_prod_workspace_min_size", "oop_debug_set_tc_schedule",
    "oop_last_launch_count", "oop_out_prod_host", "oop_out_prod_host_buffer_size",
    "oop_out_prod_plan", "oop_out_prod_strided", "oop_out_prod_strided_workspace_size",
    "oop_mul_mat_back", "oop_mul_mat_back_workspace_size",
    "oop_mul_mat_id_weight_grad", "oop_mul_mat_id_weight_grad_workspace_size",
    "oop_out_prod_batch", "oop_out_prod_batch_max", "oop_lora_backward",
)


class OopProblem(ctypes.Structure):
    """oop_out_prod_problem: one narrow single-slice OUT_PROD of a batch."""
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("dst", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("dst_transposed", ctypes.c_int)]


class OopError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if status == ERR_CUDA:
            msg += ": " + lib().oop_last_cuda_error().decode()
        super().__init__(msg)


def library_path() -> str:
    """The library file: the in-tree build, or the file named by the
    environment variable GGML_OUT_PROD_GB300_LIBRARY (e.g. a sanitizer build)."""
    return os.environ.get("GGML_OUT_PROD_GB300_LIBRARY") or _build.SO


def build(force: bool = False) -> str:
    return _build.build(force=force)


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(ggml_out_prod_gb300.build()); there is no CPU fallback")
            L = ctypes.CDLL(path)
            L.oop_out_prod_workspace_size.restype = ctypes.c_size_t
            L.oop_out_prod_workspace_size.argtypes = [ctypes.c_int, _i64p, _i64p]
            L.oop_out_prod.restype = ctypes.c_int
            L.oop_out_prod.argtypes = [_vp, ctypes.c_int, _vp, _vp, _i64p, _i64p, _i64p,
                                       _vp, ctypes.c_size_t, _vp]
            L.oop_out_prod_ex.restype = ctypes.c_int
            L.oop_out_prod_ex.argtypes = [_vp, ctypes.c_int, _vp, _vp, _i64p, _i64p, _i64p,
                                          _vp, ctypes.c_size_t, _vp, ctypes.c_int]
            L.oop_mul_mat_id_back_workspace_size.restype = ctypes.c_size_t
            L.oop_mul_mat_id_back_workspace_size.argtypes = [ctypes.c_int, _i64p, _i64p]
            L.oop_mul_mat_id_back.restype = ctypes.c_int
            L.oop_mul_mat_id_back.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _i64p, _i64p,
                                              _vp, ctypes.c_size_t, _vp]
            L.oop_mul_mat_id_back_ex.restype = ctypes.c_int
            L.oop_mul_mat_id_back_ex.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _i64p, _i64p,
                                                 _vp, ctypes.c_size_t, _vp, ctypes.c_int]
            L.oop_device_status.restype = ctypes.c_int
            L.oop_device_status.argtypes = [_vp, ctypes.c_int]
            L.oop_status_string.restype = ctypes.c_char_p
            L.oop_status_string.argtypes = [ctypes.c_int]
            L.oop_version.restype = ctypes.c_int
            L.oop_version.argtypes = []
            L.oop_out_prod_noalloc.restype = ctypes.c_int
            L.oop_out_prod_noalloc.argtypes = [_vp, ctypes.c_int, _vp, _vp, _i64p, _i64p, _i64p,
                                               _vp]
            L.oop_out_prod_noalloc_scratch_bytes.restype = ctypes.c_size_t
            L.oop_out_prod_noalloc_scratch_bytes.argtypes = []
            L.oop_profile_main_kernel.restype = ctypes.c_int
            L.oop_profile_main_kernel.argtypes = [_vp, _vp]
            L.oop_last_cuda_error.restype = ctypes.c_char_p
            L.oop_last_cuda_error.argtypes = []
            L.oop_debug_inject_timeout.restype = ctypes.c_int
            L.oop_debug_inject_timeout.argtypes = [ctypes.c_int]
            L.oop_out_prod_workspace_min_size.restype = ctypes.c_size_t
            L.oop_out_prod_workspace_min_size.argtypes = [ctypes.c_int, _i64p, _i64p]
            L.oop_debug_set_tc_schedule.restype = ctypes.c_int
            L.oop_debug_set_tc_schedule.argtypes = [ctypes.c_int]
            L.oop_last_launch_count.restype = ctypes.c_int
            L.oop_last_launch_count.argtypes = []
            L.oop_out_prod_host_buffer_size.restype = ctypes.c_size_t
            L.oop_out_prod_host_buffer_size.argtypes = [ctypes.c_int, _i64p, _i64p]
            L.oop_out_prod_host.restype = ctypes.c_int
            L.oop_out_prod_host.argtypes = [_vp, ctypes.c_int, _vp, _vp, _i64p, _i64p, _i64p,
                                            _vp, ctypes.c_size_t, _vp]
            L.oop_out_prod_plan.restype = ctypes.c_int
            L.oop_out_prod_plan.argtypes = [ctypes.c_int, _i64p, _i64p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_size_t, ctypes.POINTER(OopPlan)]
            L.oop_out_prod_strided_workspace_size.restype = ctypes.c_size_t
            L.oop_out_prod_strided_workspace_size.argtypes = [ctypes.c_int, _i64p, _i64p, _i64p]
            L.oop_out_prod_strided.restype = ctypes.c_int
            L.oop_out_prod_strided.argtypes = [_vp, ctypes.c_int, _vp, _i64p, _vp, _i64p, _i64p,
                                               _i64p, _vp, ctypes.c_size_t, _vp, ctypes.c_int]
            L.oop_mul_mat_back_workspace_size.restype = ctypes.c_size_t
            L.oop_mul_mat_back_workspace_size.argtypes = [ctypes.c_int, _i64p, _i64p]
            L.oop_mul_mat_back.restype = ctypes.c_int
            L.oop_mul_mat_back.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, _i64p, _i64p,
                                           _vp, ctypes.c_size_t, _vp]
            L.oop_mul_mat_id_weight_grad_workspace_size.restype = ctypes.c_size_t
            L.oop_mul_mat_id_weight_grad_workspace_size.argtypes = [_i64p, _i64p, ctypes.c_int64]
            L.oop_mul_mat_id_weight_grad.restype = ctypes.c_int
            L.oop_mul_mat_id_weight_grad.argtypes = [_vp, _vp, _vp, _vp, _i64p, _i64p,
                                                     ctypes.c_int64, _vp, ctypes.c_size_t, _vp]
            L.oop_out_prod_batch_max.restype = ctypes.c_int
            L.oop_out_prod_batch_max.argtypes = []
            L.oop_out_prod_batch.restype = ctypes.c_int
            L.oop_out_prod_batch.argtypes = [ctypes.POINTER(OopProblem), ctypes.c_int,
                                             ctypes.c_int64, _vp]
            L.oop_lora_backward.restype = ctypes.c_int
            L.oop_lora_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _vp]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().oop_status_string(int(status)).decode()


def _ne(v):
    v = list(v)
    return (ctypes.c_int64 * len(v))(*[int(x) for x in v])


# ---------------------------------------------------------------------------
# C-ABI mirrors (plain pointers and sizes)
# ---------------------------------------------------------------------------

def oop_out_prod_workspace_size(a_type, ne_a, ne_b) -> int:
    return int(lib().oop_out_prod_workspace_size(int(a_type), _ne(ne_a), _ne(ne_b)))


class OopPlan(ctypes.Structure):
    """oop_plan: the kernels an OUT_PROD call would enqueue."""
    _fields_ = [("path", ctypes.c_int), ("kernel", ctypes.c_int), ("item_m", ctypes.c_int),
                ("ctas", ctypes.c_int), ("launches", ctypes.c_int)]


KERNEL_NONE, KERNEL_SKINNY, KERNEL_SKINNY_TMA = 0, 1, 2
KERNEL_TC_DATA_PARALLEL, KERNEL_TC_STREAM_K, KERNEL_SIMT = 3, 4, 5


def oop_out_prod_plan(a_type, ne_a, ne_b, path, sms, workspace_bytes):
    """(status, OopPlan) from the library's planner; no device is needed."""
    plan = OopPlan()
    rc = lib().oop_out_prod_plan(int(a_type), _ne(ne_a), _ne(ne_b), int(path), int(sms),
                                 int(workspace_bytes), ctypes.byref(plan))
    return int(rc), plan


def out_prod_plan(a_type, ne_a, ne_b, sms, path=0, workspace_bytes=None) -> dict:
    """The plan of an OUT_PROD call on a GPU with `sms` SMs (default workspace:
    oop_out_prod_workspace_size); raises OopError on an argument error."""
    if workspace_bytes is None:
        workspace_bytes = oop_out_prod_workspace_size(a_type, ne_a, ne_b)
    rc, p = oop_out_prod_plan(a_type, ne_a, ne_b, path, sms, workspace_bytes)
    if rc != 0:
        raise OopError(rc, "oop_out_prod_plan")
    return {"path": p.path, "kernel": p.kernel, "item_m": p.item_m, "ctas": p.ctas,
            "launches": p.launches}


def oop_out_prod_workspace_min_size(a_type, ne_a, ne_b) -> int:
    return int(lib().oop_out_prod_workspace_min_size(int(a_type), _ne(ne_a), _ne(ne_b)))


def oop_debug_set_tc_schedule(mode) -> int:
    return int(lib().oop_debug_set_tc_schedule(int(mode)))


def oop_last_launch_count() -> int:
    return int(lib().oop_last_launch_count())


def oop_out_prod_host_buffer_size(a_type, ne_a, ne_b) -> int:
    return int(lib().oop_out_prod_host_buffer_size(int(a_type), _ne(ne_a), _ne(ne_b)))


def oop_out_prod_host(a, a_type, b, dst, ne_a, ne_b, ne_dst, device_buffer, device_bytes,
                      stream) -> int:
    return int(lib().oop_out_prod_host(a, int(a_type), b, dst, _ne(ne_a), _ne(ne_b), _ne(ne_dst),
                                       device_buffer, int(device_bytes), stream))


def oop_out_prod(a, a_type, b, dst, ne_a, ne_b, ne_dst, workspace, workspace_bytes, stream,
                 path=PATH_AUTO) -> int:
    return int(lib().oop_out_prod_ex(a, int(a_type), b, dst, _ne(ne_a), _ne(ne_b), _ne(ne_dst),
                                     workspace, int(workspace_bytes), stream, int(path)))


def oop_out_prod_noalloc(a, a_type, b, dst, ne_a, ne_b, ne_dst, stream) -> int:
    """OUT_PROD with the library's own fixed device scratch (no allocation)."""
    return int(lib().oop_out_prod_noalloc(a, int(a_type), b, dst, _ne(ne_a), _ne(ne_b),
                                          _ne(ne_dst), stream))


def oop_out_prod_strided_workspace_size(a_type, ne_a, ne_b, nb_b) -> int:
    return int(lib().oop_out_prod_strided_workspace_size(int(a_type), _ne(ne_a), _ne(ne_b),
                                                         _ne(nb_b)))


def oop_out_prod_strided(a, a_type, b, nb_b, dst, ne_a, ne_b, ne_dst, workspace,
                         workspace_bytes, stream, path=PATH_AUTO) -> int:
    return int(lib().oop_out_prod_strided(a, int(a_type), b, _ne(nb_b), dst, _ne(ne_a),
                                          _ne(ne_b), _ne(ne_dst), workspace,
                                          int(workspace_bytes), stream, int(path)))


def oop_mul_mat_back_workspace_size(w_type, ne_w, ne_x) -> int:
    return int(lib().oop_mul_mat_back_workspace_size(int(w_type), _ne(ne_w), _ne(ne_x)))


def oop_mul_mat_back(W, w_type, x, dy, dW, dx, ne_w, ne_x, workspace, workspace_bytes,
                     stream) -> int:
    return int(lib().oop_mul_mat_back(W, int(w_type), x, dy, dW, dx, _ne(ne_w), _ne(ne_x),
                                      workspace, int(workspace_bytes), stream))


def oop_mul_mat_id_weight_grad_workspace_size(ne_x, ne_dy, n_expert) -> int:
    return int(lib().oop_mul_mat_id_weight_grad_workspace_size(_ne(ne_x), _ne(ne_dy),
                                                               int(n_expert)))


def oop_mul_mat_id_weight_grad(x, ids, dy, dW, ne_x, ne_dy, n_expert, workspace,
                               workspace_bytes, stream) -> int:
    return int(lib().oop_mul_mat_id_weight_grad(x, ids, dy, dW, _ne(ne_x), _ne(ne_dy),
                                                int(n_expert), workspace, int(workspace_bytes),
                                                stream))


def oop_mul_mat_id_back_workspace_size(w_type, ne_w, ne_ids) -> int:
    return int(lib().oop_mul_mat_id_back_workspace_size(int(w_type), _ne(ne_w), _ne(ne_ids)))


def oop_mul_mat_id_back(W, w_type, ids, g, dx, ne_w, ne_ids, workspace, workspace_bytes,
                        stream, path=PATH_AUTO) -> int:
    return int(lib().oop_mul_mat_id_back_ex(W, int(w_type), ids, g, dx, _ne(ne_w), _ne(ne_ids),
                                            workspace, int(workspace_bytes), stream, int(path)))


def oop_device_status(stream=None, clear=True) -> int:
    return int(lib().oop_device_status(stream, 1 if clear else 0))


# ---------------------------------------------------------------------------
# torch-level convenience (argument marshalling only)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None


def ne_of(t, type_id=TYPE_F32, ne0=None):
    """ggml ne of a contiguous tensor in this layout (a quantised src0's last
    axis holds one row's block bytes)."""
    shp = (1,) * (4 - t.dim()) + tuple(t.shape)
    if type_id in _BLOCKS:
        if ne0 is None:
            qk, nbytes = _BLOCKS[type_id]
            ne0 = shp[3] // nbytes * qk
        return (ne0, shp[2], shp[1], shp[0])
    return (shp[3], shp[2], shp[1], shp[0])


def _check_src0(t, type_id, name):
    torch = _torch()
    if type_id == TYPE_F32 and t.dtype != torch.float32:
        raise ValueError(f"f32 {name} must be a float32 tensor")
    if type_id in _HALF_TYPES and t.element_size() != 2:
        raise ValueError(f"f16 / bf16 {name} must hold 2-byte elements")
    if type_id in _BLOCKS and t.dtype != torch.uint8:
        raise ValueError(f"quantised {name} must be a uint8 tensor of block bytes")


def _check_cuda(t, name, contiguous=True):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def nb_of(t):
    """ggml byte strides nb of a float32 tensor view in this layout."""
    st = (0,) * (4 - t.dim()) + tuple(t.stride())
    if any(x < 0 for x in st):
        raise ValueError("negative strides are not supported")
    return (4 * st[3], 4 * st[2], 4 * st[1], 4 * st[0])


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if nbytes == 0:
        return None
    if workspace is not None:
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def out_prod(a, b, a_type=None, ne_a=None, out=None, workspace=None, stream=None,
             path=PATH_AUTO):
    """dst = OUT_PROD(a, b) on a's device and the current (or given) stream.

    a: float32 tensor, a tensor of 2-byte f16 / bf16 elements, or uint8 rows of
    quantised blocks (give ``a_type``); b: float32,
    contiguous or any view with non-negative strides (a transpose, a slice),
    which is read in place through oop_out_prod_strided.
    Returns dst, float32 of shape (ne13, ne12, N, M)."""
    torch = _torch()
    if a_type is None:
        a_type = TYPE_F32
    _check_cuda(a, "a")
    _check_cuda(b, "b", contiguous=False)
    if b.dtype != torch.float32:
        raise ValueError("b must be float32")
    _check_src0(a, a_type, "src0")
    if ne_a is None:
        ne_a = ne_of(a, a_type)
    ne_b = ne_of(b)
    ne_dst = (ne_a[0], ne_b[0], ne_b[2], ne_b[3])
    if out is None:
        out = torch.empty((ne_dst[3], ne_dst[2], ne_dst[1], ne_dst[0]), dtype=torch.float32,
                          device=a.device)
    _check_cuda(out, "out")
    if b.is_contiguous():
        nws = oop_out_prod_workspace_size(a_type, ne_a, ne_b)
        ws = _workspace(nws, a.device, workspace)
        rc = oop_out_prod(_ptr(a), a_type, _ptr(b), _ptr(out), ne_a, ne_b, ne_dst, _ptr(ws),
                          ws.numel() if ws is not None else 0, _stream_ptr(stream), path)
        if rc != OK:
            raise OopError(rc, "oop_out_prod")
        return out
    nb_b = nb_of(b)
    nws = oop_out_prod_strided_workspace_size(a_type, ne_a, ne_b, nb_b)
    ws = _workspace(nws, a.device, workspace)
    rc = oop_out_prod_strided(_ptr(a), a_type, _ptr(b), nb_b, _ptr(out), ne_a, ne_b, ne_dst,
                              _ptr(ws), ws.numel() if ws is not None else 0,
                              _stream_ptr(stream), path)
    if rc != OK:
        raise OopError(rc, "oop_out_prod_strided")
    return out


def mul_mat_back(W, x, dy, w_type=None, ne_w=None, want_dW=True, want_dx=True,
                 workspace=None, stream=None):
    """Both gradients of y = MUL_MAT(W, x) from dy, in one call.

    W: float32 (ne03, ne02, R, K), or uint8 q8_0/q4_0 rows (give ``w_type``
    and ``ne_w``); x: float32 (ne13, ne12, T, K); dy: float32
    (ne13, ne12, T, R).  Returns (dW, dx): dW float32 (ne03, ne02, R, K) or
    None, dx float32 like x or None."""
    torch = _torch()
    if w_type is None:
        w_type = TYPE_F32
    for t, n in ((W, "W"), (x, "x"), (dy, "dy")):
        _check_cuda(t, n)
    if x.dtype != torch.float32 or dy.dtype != torch.float32:
        raise ValueError("x and dy must be float32")
    _check_src0(W, w_type, "W")
    if ne_w is None:
        ne_w = ne_of(W, w_type)
    ne_x = ne_of(x)
    dW = torch.empty((ne_w[3], ne_w[2], ne_w[1], ne_w[0]), dtype=torch.float32,
                     device=W.device) if want_dW else None
    dx = torch.empty_like(x) if want_dx else None
    nws = oop_mul_mat_back_workspace_size(w_type, ne_w, ne_x)
    ws = _workspace(nws, W.device, workspace)
    rc = oop_mul_mat_back(_ptr(W), w_type, _ptr(x), _ptr(dy), _ptr(dW), _ptr(dx), ne_w, ne_x,
                          _ptr(ws), ws.numel() if ws is not None else 0, _stream_ptr(stream))
    if rc != OK:
        raise OopError(rc, "oop_mul_mat_back")
    return dW, dx


def mul_mat_id_back(W, ids, g, w_type=None, out=None, workspace=None, stream=None,
                    path=PATH_AUTO, K=None):
    """dx = MUL_MAT_ID_BACK(W, ids, g).

    W: float32 (E, N, K), 2-byte f16 / bf16 elements (E, N, K), or uint8
    rows of quantised blocks (E, N, row bytes; give ``w_type``, K is derived
    from the row bytes unless given); ids: int32 (n_tokens, n_used); g: float32
    (n_tokens, n_used, N).  Returns dx float32 (n_tokens, n_used, K)."""
    torch = _torch()
    for t, n in ((W, "W"), (ids, "ids"), (g, "g")):
        _check_cuda(t, n)
    if w_type is None:
        w_type = TYPE_F32 if W.dtype == torch.float32 else TYPE_BF16
    _check_src0(W, w_type, "W")
    if ids.dtype != torch.int32 or g.dtype != torch.float32:
        raise ValueError("ids must be int32 and g float32")
    E, N, K_row = W.shape
    if K is None:
        K = K_row // _BLOCKS[w_type][1] * _BLOCKS[w_type][0] if w_type in _BLOCKS else K_row
    n_tok, n_used = ids.shape
    if tuple(g.shape) != (n_tok, n_used, N):
        raise ValueError("g must be (n_tokens, n_used, N)")
    if out is None:
        out = torch.empty((n_tok, n_used, K), dtype=torch.float32, device=W.device)
    _check_cuda(out, "out")
    ne_w, ne_ids = (K, N, E), (n_used, n_tok)
    nws = oop_mul_mat_id_back_workspace_size(w_type, ne_w, ne_ids)
    ws = _workspace(nws, W.device, workspace)
    rc = oop_mul_mat_id_back(_ptr(W), w_type, _ptr(ids), _ptr(g), _ptr(out), ne_w, ne_ids,
                             _ptr(ws), ws.numel() if ws is not None else 0,
                             _stream_ptr(stream), path)
    if rc != OK:
        raise OopError(rc, "oop_mul_mat_id_back")
    return out


def mul_mat_id_weight_grad(x, ids, dy, n_expert, out=None, workspace=None, stream=None):
    """dW = the expert-weight gradient of MUL_MAT_ID.

    x: float32 (n_tokens, n_x, K); ids: int32 (n_tokens, n_used); dy: float32
    (n_tokens, n_used, N).  Returns dW float32 (n_expert, N, K)."""
    torch = _torch()
    for t, n in ((x, "x"), (ids, "ids"), (dy, "dy")):
        _check_cuda(t, n)
    if x.dtype != torch.float32 or dy.dtype != torch.float32 or ids.dtype != torch.int32:
        raise ValueError("x and dy must be float32, ids int32")
    n_tok, n_x, K = x.shape
    _, n_used, N = dy.shape
    ne_x, ne_dy = (K, n_x, n_tok), (N, n_used, n_tok)
    if out is None:
        out = torch.empty((n_expert, N, K), dtype=torch.float32, device=x.device)
    _check_cuda(out, "out")
    nws = oop_mul_mat_id_weight_grad_workspace_size(ne_x, ne_dy, n_expert)
    ws = _workspace(nws, x.device, workspace)
    rc = oop_mul_mat_id_weight_grad(_ptr(x), _ptr(ids), _ptr(dy), _ptr(out), ne_x, ne_dy,
                                    n_expert, _ptr(ws), ws.numel() if ws is not None else 0,
                                    _stream_ptr(stream))
    if rc != OK:
        raise OopError(rc, "oop_mul_mat_id_weight_grad")
    return out


def oop_out_prod_batch(problems, N, stream) -> int:
    """problems: a sequence of OopProblem (or (a, b, dst, M, K, transposed) tuples of
    device pointers and sizes)."""
    arr = (OopProblem * max(len(problems), 1))()
    for i, q in enumerate(problems):
        arr[i] = q if isinstance(q, OopProblem) else OopProblem(*q)
    return int(lib().oop_out_prod_batch(arr, len(problems), int(N), stream))


def out_prod_batch(problems, stream=None):
    """Narrow OUT_PRODs in one call: ``problems`` is a list of (a, b, dst) or
    (a, b, dst, transposed) torch float32 CUDA tensors with a (K, M), b (K, N)
    and dst (N, M) -- or (M, N) when transposed -- and one N for all."""
    if not problems:
        return
    Ns = {q[1].shape[-1] for q in problems}
    if len(Ns) != 1:
        raise ValueError("every problem of a batch has the same N")
    N = Ns.pop()
    items = []
    for q in problems:
        a, b, dst = q[0], q[1], q[2]
        tr = bool(q[3]) if len(q) > 3 else False
        for t, n in ((a, "a"), (b, "b"), (dst, "dst")):
            _check_cuda(t, n)
        K, M = a.shape[-2], a.shape[-1]
        if b.shape[-2] != K or tuple(dst.shape[-2:]) != ((M, N) if tr else (N, M)):
            raise ValueError("shapes do not match")
        items.append(OopProblem(a.data_ptr() if a.numel() else None,
                                b.data_ptr() if b.numel() else None, dst.data_ptr(), M, K,
                                1 if tr else 0))
    rc = oop_out_prod_batch(items, N, _stream_ptr(stream))
    if rc != OK:
        raise OopError(rc, "oop_out_prod_batch")


def lora_backward(x, h, dz, dh, stream=None):
    """Both LoRA adapter gradients of one projection in one launch.

    x (T, K_in), h (T, r), dz (T, N_out), dh (T, r): float32 CUDA tensors
    (ggml {K_in, T}, {r, T}, {N_out, T}, {r, T}).  Returns (dA, dB): dA
    (r, K_in) = ggml {K_in, r}, dB (N_out, r) = ggml {r, N_out}."""
    torch = _torch()
    for t, n in ((x, "x"), (h, "h"), (dz, "dz"), (dh, "dh")):
        _check_cuda(t, n)
    T, K_in = x.shape
    r = h.shape[1]
    N_out = dz.shape[1]
    dA = torch.empty((r, K_in), dtype=torch.float32, device=x.device)
    dB = torch.empty((N_out, r), dtype=torch.float32, device=x.device)
    rc = int(lib().oop_lora_backward(_ptr(x), _ptr(h), _ptr(dz), _ptr(dh), _ptr(dA), _ptr(dB),
                                     K_in, N_out, T, r, _stream_ptr(stream)))
    if rc != OK:
        raise OopError(rc, "oop_lora_backward")
    return dA, dB


def profile_main_kernel(before, after) -> None:
    """Have the next tensor-core launch record torch.cuda.Event `before` and
    `after` around its main tile kernel (the events must exist already:
    record each once first)."""
    lib().oop_profile_main_kernel(ctypes.c_void_p(before.cuda_event),
                                  ctypes.c_void_p(after.cuda_event))


def device_status(stream=None, clear=True) -> int:
    return oop_device_status(_stream_ptr(stream), clear)


def set_tc_schedule(mode) -> None:
    """Pick the tensor-core tile kernel's schedule for the calls that follow
    (SCHEDULE_AUTO, SCHEDULE_DATA_PARALLEL or SCHEDULE_STREAM_K)."""
    rc = oop_debug_set_tc_schedule(mode)
    if rc != OK:
        raise OopError(rc, "oop_debug_set_tc_schedule")


def last_launch_count() -> int:
    """Kernels the last OUT_PROD / MUL_MAT_ID_BACK call on this thread enqueued."""
    return oop_last_launch_count()


def out_prod_host(a_host, b_host, a_type=None, ne_a=None, out=None, device_buffer=None,
                  stream=None):
    """OUT_PROD from host tensors through the C ABI's host entry: the copies
    in, the product and the copy of dst out are enqueued by one call (up to
    four chunks of k pipelined when the shape allows), then the stream is
    synchronised.  a_host / b_host: CPU tensors (pinned memory makes the
    copies asynchronous); ``out``: a CPU float32 tensor of dst's shape
    (allocated pinned when None); ``device_buffer``: a CUDA uint8 tensor of at
    least oop_out_prod_host_buffer_size bytes (allocated when None)."""
    torch = _torch()
    if a_type is None:
        a_type = TYPE_F32
    for t, n in ((a_host, "a_host"), (b_host, "b_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    if b_host.dtype != torch.float32:
        raise ValueError("b_host must be float32")
    if ne_a is None:
        ne_a = ne_of(a_host, a_type)
    ne_b = ne_of(b_host)
    ne_dst = (ne_a[0], ne_b[0], ne_b[2], ne_b[3])
    if out is None:
        out = torch.empty((ne_dst[3], ne_dst[2], ne_dst[1], ne_dst[0]), dtype=torch.float32,
                          pin_memory=True)
    nbuf = oop_out_prod_host_buffer_size(a_type, ne_a, ne_b)
    if device_buffer is None:
        device_buffer = torch.empty(max(nbuf, 1), dtype=torch.uint8, device="cuda")
    st = _stream_ptr(stream)
    rc = oop_out_prod_host(_ptr(a_host), a_type, _ptr(b_host), _ptr(out), ne_a, ne_b, ne_dst,
                           _ptr(device_buffer), device_buffer.numel(), st)
    if rc != OK:
        raise OopError(rc, "oop_out_prod_host")
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return out
