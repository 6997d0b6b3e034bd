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
from helpers import TOL, assert_parity, sample_coords

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


def test_no_alloc_skinny_needs_no_scratch(op, orc):
    """f32 src0 with N <= 32 runs on the skinny-N kernel, which needs no
    scratch, even where the tensor-core kernel's split of this gradient
    (84 MiB here) would not fit in the array."""
    import torch
    cap = op.lib().oop_out_prod_noalloc_scratch_bytes()
    ne_a, ne_b = (64, 8192, 1, 1), (32, 8192, 40, 1)
    assert op.oop_out_prod_workspace_min_size(op.TYPE_F32, ne_a, ne_b) > cap
    a = synth.make_a(op.TYPE_F32, ne_a, 82)
    b = synth.make_b(ne_b, 83, std=100.0, outliers=True)
    exact = orc.out_prod(a, op.TYPE_F32, b, ne_a, ne_b)
    for _ in range(2):
        ref, got = _call_both(op, torch, a, op.TYPE_F32, b, ne_a, ne_b)
        assert_parity(got, exact["f64"], exact["abs"], "no-alloc skinny")
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_no_alloc_minimum_fits_full_does_not(op, orc):
    """The tensor-core minimum (the split, 56 MiB) fits in the array but the
    stream-K partials on top of it do not: the call runs the data-parallel
    schedule, allocates nothing (device memory in use is unchanged across a
    repeated call) and matches the oracle on sampled elements."""
    import torch
    cap = op.lib().oop_out_prod_noalloc_scratch_bytes()
    M, K, N = 256, 7168, 1024
    ne_a, ne_b = (M, K, 1, 1), (N, K, 1, 1)
    assert op.oop_out_prod_workspace_min_size(synth.TYPE_Q8_0, ne_a, ne_b) <= cap
    assert op.oop_out_prod_workspace_size(synth.TYPE_Q8_0, ne_a, ne_b) > cap
    a = synth.make_a(synth.TYPE_Q8_0, ne_a, 84, std=0.02)
    b = synth.make_b(ne_b, 85, std=1e3, outliers=True)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = torch.full((1, 1, N, M), float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        rc = op.oop_out_prod_noalloc(_ptr(ta), synth.TYPE_Q8_0, _ptr(tb), _ptr(out), ne_a, ne_b,
                                     (M, N, 1, 1), stream)
        assert rc == op.OK, op.status_string(rc)

    call()                                  # first call: address look-up, module load
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory in use changed by {free0 - free1} bytes"
    assert op.device_status() == op.OK
    rng = np.random.default_rng(86)
    coords = sample_coords(rng, (M, N, 1, 1), 2000)
    val, ab = orc.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords)
    got = out.cpu().numpy()[coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]]
    assert_parity(got, val, ab, "no-alloc, data-parallel within the array")
