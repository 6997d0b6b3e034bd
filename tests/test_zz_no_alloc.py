"""The allocation-free OUT_PROD entry point, through the C ABI.

Some callers cannot allocate device memory (a framework allocator that owns
all of it, plug-ins given fixed tensors, loops where cudaMalloc would
synchronise the device).  oop_out_prod_noalloc uses the library's own fixed
device scratch instead of a caller workspace.  This file is collected last so
that a failure here leaves every other test already run; it passes on its own
in a fresh process as well.
"""

import ctypes

import numpy as np
import pytest

import synth
from helpers import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_both(op, torch, a, a_type, b, ne_a, ne_b):
    ne_dst = (ne_a[0], ne_b[0], ne_b[2], ne_b[3])
    shape = (ne_dst[3], ne_dst[2], ne_dst[1], ne_dst[0])
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # existing entry point, caller-provided workspace
    ref = torch.full(shape, float("nan"), device="cuda")
    nws = op.oop_out_prod_workspace_size(a_type, ne_a, ne_b)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
    rc = op.oop_out_prod(_ptr(ta), a_type, _ptr(tb), _ptr(ref), ne_a, ne_b, ne_dst,
                         _ptr(ws), nws, stream)
    assert rc == op.OK
    # the allocation-free entry point
    got = torch.full(shape, float("nan"), device="cuda")
    rc = op.oop_out_prod_noalloc(_ptr(ta), a_type, _ptr(tb), _ptr(got), ne_a, ne_b, ne_dst,
                                 stream)
    assert rc == op.OK, op.status_string(rc)
    torch.cuda.synchronize()
    assert op.device_status() == op.OK
    return ref.cpu().numpy(), got.cpu().numpy()


def test_no_alloc_matches_workspace_entry_two_calls(op, orc):
    import torch
    calls = [
        (synth.TYPE_Q8_0, (1536, 1536, 1, 1), (1024, 1536, 1, 1), 0.02, 1e3),
        (synth.TYPE_F32, (128, 512, 4, 2), (128, 512, 16, 2), 1.0, 1.0),
    ]
    for a_type, ne_a, ne_b, sa, sb in calls:
        a = synth.make_a(a_type, ne_a, 80, std=sa)
        b = synth.make_b(ne_b, 81, std=sb, outliers=True)
        assert op.oop_out_prod_workspace_size(a_type, ne_a, ne_b) <= \
            op.lib().oop_out_prod_noalloc_scratch_bytes()
        ref, got = _call_both(op, torch, a, a_type, b, ne_a, ne_b)
        exact = orc.out_prod(a, a_type, b, ne_a, ne_b)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got.astype(np.float64) - ref) <= TOL * exact["abs"])
        assert np.all(np.abs(got.astype(np.float64) - exact["f64"]) <= TOL * exact["abs"])


def test_no_alloc_rejects_too_much_scratch(op):
    import torch
    cap = op.lib().oop_out_prod_noalloc_scratch_bytes()
    ne_a, ne_b = (256, 8192, 1, 1), (2048, 8192, 1, 1)       # 128 MiB of split gradient
    assert op.oop_out_prod_workspace_size(op.TYPE_F32, ne_a, ne_b) > cap
    dummy = torch.empty(16, device="cuda")
    rc = op.oop_out_prod_noalloc(_ptr(dummy), op.TYPE_F32, _ptr(dummy), _ptr(dummy), ne_a,
                                 ne_b, (256, 2048, 1, 1), None)
    assert rc == op.ERR_SCRATCH_LIMIT
    assert "scratch" in op.status_string(rc)
