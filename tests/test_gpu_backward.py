"""GPU parity of OUT_PROD with a strided src1 view and of the MUL_MAT
backward pair, against the CPU oracle, through the C ABI.

The gradient of a MUL_MAT's src1 is out_prod(src0, grad^T) ("metal: OUT_PROD
multiplies in float staging; a training gradient overflowed half", scope
paragraph); the view lets grad^T be read in place.  Every case checks, element
by element, |gpu - exact| <= 2e-6 * sum_k |a*b| and zero non-finite outputs.
"""

import numpy as np
import pytest

import synth
from helpers import assert_parity, sample_coords

pytestmark = pytest.mark.gpu

F32, Q8, Q4 = synth.TYPE_F32, synth.TYPE_Q8_0, synth.TYPE_Q4_0


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


def _views(N, K, S2, S3, seed):
    """(name, numpy view of shape (S3, S2, K, N), the same view on the device)
    triples, each a view of one base array with the same strides."""
    import torch
    tr = synth.make_b((K, N, S2, S3), seed, std=1e3, outliers=True)     # (S3, S2, N, K)
    pad = synth.make_b((N + 5, K, S2, S3), seed + 1, std=1e3, outliers=True)
    step = synth.make_b((N, K, 2 * S2, S3), seed + 2, std=1e3, outliers=True)
    row = synth.make_b((1, K, S2, S3), seed + 3, std=1e3, outliers=True)
    d = {k: torch.from_numpy(v).cuda() for k, v in
         (("tr", tr), ("pad", pad), ("step", step), ("row", row))}
    return [
        ("transposed (k contiguous)", np.swapaxes(tr, 2, 3), d["tr"].transpose(2, 3)),
        ("padded rows", pad[:, :, :, 2:2 + N], d["pad"][:, :, :, 2:2 + N]),
        ("every other slice", step[:, ::2], d["step"][:, ::2]),
        ("one row for every n (zero stride)", np.broadcast_to(row, (S3, S2, K, N)),
         d["row"].expand(S3, S2, K, N)),
    ]


def _paths(op, a_type, N):
    ps = [op.PATH_AUTO, op.PATH_TCGEN05, op.PATH_SIMT]
    if a_type == F32 and N <= 32:
        ps.append(op.PATH_SKINNY)
    return ps


@pytest.mark.parametrize("a_type,M,N,K,S2,S3,A2,A3", [
    (F32, 160, 200, 300, 2, 1, 1, 1),      # dense side, several tiles, ragged n and k
    (F32, 130, 24, 257, 2, 2, 2, 1),       # skinny side, broadcast
    (Q8, 256, 100, 200, 3, 1, 3, 1),
    (Q4, 192, 130, 96, 1, 2, 1, 1),
])
def test_strided_views(op, orc, a_type, M, N, K, S2, S3, A2, A3):
    import torch
    ne_a = (M, K, A2, A3)
    a = synth.make_a(a_type, ne_a, 130, std=0.02 if a_type != F32 else 1.0)
    ta = torch.from_numpy(a).cuda()
    for name, v, tv in _views(N, K, S2, S3, 131):
        ref = orc.out_prod_strided(a, a_type, v, ne_a)
        assert not tv.is_contiguous() and tuple(tv.shape) == v.shape
        assert all(4 * t == n for t, n, d in zip(tv.stride(), v.strides, v.shape) if d > 1)
        for p in _paths(op, a_type, N):
            out = op.out_prod(ta, tv, a_type=a_type, ne_a=ne_a, path=p)
            torch.cuda.synchronize()
            assert op.device_status() == 0
            assert_parity(out.cpu().numpy(), ref["f64"], ref["abs"], f"{name} path {p}")


def test_transposed_gradient_full_size_sampled(op, orc):
    """dx of the dense training shape through the view: W q8_0 [5120, 5120],
    dy [5120, 1024] read as dy^T; sampled elements against the oracle."""
    import torch
    K, R, T = 5120, 5120, 1024
    W = synth.make_a(Q8, (K, R, 1, 1), 132, std=0.02)
    dy = synth.make_b((R, T, 1, 1), 133, std=1e3, outliers=True)       # (1, 1, T, R)
    tW, tdy = torch.from_numpy(W).cuda(), torch.from_numpy(dy).cuda()
    dyT = tdy.transpose(2, 3)                                          # (1, 1, R, T) view
    out = op.out_prod(tW, dyT, a_type=Q8, ne_a=(K, R, 1, 1))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(134)
    coords = sample_coords(rng, (K, T, 1, 1), 1500)
    val, ab = orc.out_prod_at(W, Q8, np.ascontiguousarray(np.swapaxes(dy, 2, 3)),
                              (K, R, 1, 1), (T, R, 1, 1), coords)
    got = out.cpu().numpy()[coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]]
    assert_parity(got, val, ab, "dx through the transposed view, full size")


@pytest.mark.parametrize("w_type", [F32, Q8, Q4])
@pytest.mark.parametrize("ne_w,ne_x", [
    ((256, 100, 1, 1), (256, 70, 1, 1)),        # dense dx and dW
    ((160, 24, 1, 1), (160, 20, 1, 1)),         # narrow: skinny dW, skinny dx (f32 W)
    ((128, 96, 2, 1), (128, 40, 6, 1)),         # dps2 = 3: dW sums adjacent slices
    ((96, 48, 1, 2), (96, 33, 3, 4)),           # ne02 = 1, dps3 = 2
])
def test_mul_mat_back_pair(op, orc, w_type, ne_w, ne_x):
    import torch
    K, R, w2, w3 = ne_w
    _, T, x2, x3 = ne_x
    W = synth.make_a(w_type, ne_w, 135, std=0.02 if w_type != F32 else 1.0)
    x = synth.make_b((K, T, x2, x3), 136)
    dy = synth.make_b((R, T, x2, x3), 137, std=1e3, outliers=True)
    ref = orc.mul_mat_back(W, w_type, x, dy, ne_w)
    tW, tx, tdy = (torch.from_numpy(v).cuda() for v in (W, x, dy))
    for want_dW, want_dx in ((True, True), (False, True), (True, False)):
        dW, dx = op.mul_mat_back(tW, tx, tdy, w_type=w_type, ne_w=ne_w, want_dW=want_dW,
                                 want_dx=want_dx)
        torch.cuda.synchronize()
        assert op.device_status() == 0
        if want_dx:
            assert_parity(dx.cpu().numpy(), ref["dx"]["f64"], ref["dx"]["abs"], "dx")
        if want_dW:
            assert_parity(dW.cpu().numpy(), ref["dW"]["f64"], ref["dW"]["abs"], "dW")


def test_mul_mat_back_rejects_before_enqueueing(op):
    """dW over broadcast groups that are not adjacent in memory (dps3 > 1 with
    ne02 > 1) is refused before anything runs: dx is left untouched too."""
    import torch
    ne_w, ne_x = (64, 16, 2, 1), (64, 8, 4, 2)
    W = torch.ones((1, 2, 16, 64), device="cuda")
    x = torch.ones((2, 4, 8, 64), device="cuda")
    dy = torch.ones((2, 4, 8, 16), device="cuda")
    dW = torch.full((1, 2, 16, 64), 7.0, device="cuda")
    dx = torch.full((2, 4, 8, 64), 7.0, device="cuda")
    nws = op.oop_mul_mat_back_workspace_size(F32, ne_w, ne_x)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())     # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # ne13 = 2 over ne03 = 1: dps3 = 2 with ne02 = 2
    rc = op.oop_mul_mat_back(p(W), F32, p(x), p(dy), p(dW), p(dx), ne_w, (64, 8, 4, 2),
                             p(ws), nws, stream)
    assert rc == op.ERR_BROADCAST
    torch.cuda.synchronize()
    assert bool((dx == 7.0).all()) and bool((dW == 7.0).all())
    # without dW the same call is fine
    rc = op.oop_mul_mat_back(p(W), F32, p(x), p(dy), None, p(dx), ne_w, (64, 8, 4, 2),
                             p(ws), nws, stream)
    assert rc == op.OK
    torch.cuda.synchronize()
    assert bool((dx == 16.0).all())
