"""fp32's range at both ends, on every kernel, against the CPU oracle.

Every finite input must give a finite result inside 2e-6 * sum_k |a*b| of
the exact sum ("metal: OUT_PROD multiplies in float staging; a training
gradient overflowed half", opening paragraph: a staging format that lost
range turned finite gradients into Inf).  The tensor-core kernels split each
operand into two TF32 terms; these cases reach the top binade of fp32 (where
rounding to nearest would carry into the exponent), products and sums in the
subnormal range, and the extreme binary16 block scales of q8_0 / q4_0
weights.
"""

import numpy as np
import pytest

import synth
from helpers import assert_parity

pytestmark = pytest.mark.gpu

F32, Q8, Q4 = synth.TYPE_F32, synth.TYPE_Q8_0, synth.TYPE_Q4_0
FLT_MAX = float(np.finfo(np.float32).max)
# the smallest magnitude whose round-to-nearest TF32 value would be 2^128
TOP_CARRY = float(np.uint32(0x7F7FF000).view(np.float32))


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


def _paths(op, a_type, N):
    ps = [op.PATH_AUTO, op.PATH_TCGEN05, op.PATH_SIMT]
    if a_type == F32 and N <= 32:
        ps.append(op.PATH_SKINNY)
    return ps


def _run(op, a, a_type, b, ne_a, path):
    import torch
    ta = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tb = torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).cuda()
    out = op.out_prod(ta, tb, a_type=a_type, ne_a=ne_a, path=path)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    return out.cpu().numpy()


def _check(op, orc, a, a_type, b, ne_a, ne_b, what, terms=0):
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    assert np.all(np.isfinite(ref["f64"])), "the case itself must have a finite result"
    for p in _paths(op, a_type, ne_b[0]):
        for sched in (op.SCHEDULE_AUTO, op.SCHEDULE_STREAM_K):
            if sched != op.SCHEDULE_AUTO and p not in (op.PATH_TCGEN05, op.PATH_AUTO):
                continue
            op.set_tc_schedule(sched)
            try:
                got = _run(op, a, a_type, b, ne_a, p)
            finally:
                op.set_tc_schedule(op.SCHEDULE_AUTO)
            assert_parity(got, ref["f64"], ref["abs"], f"{what} path {p} schedule {sched}",
                          terms=terms)


def _plant(x, rng, values, count):
    """Overwrite `count` random entries of x with entries drawn from values."""
    flat = x.reshape(-1)
    idx = rng.choice(flat.size, size=count, replace=False)
    flat[idx] = rng.choice(np.asarray(values, dtype=np.float32), size=count)
    return x


TOP = [FLT_MAX, -FLT_MAX, TOP_CARRY, -TOP_CARRY,
       float(np.uint32(0x7F7FFFFE).view(np.float32)), float(np.uint32(0xFF7FF800).view(np.float32))]


@pytest.mark.parametrize("N", [100, 24])
def test_top_binade_in_src0(op, orc, N):
    """a holds values at and next to FLT_MAX, b ~ 1e-30: products ~3e8."""
    rng = np.random.default_rng(1)
    M, K = 160, 72
    a = synth.make_a(F32, (M, K, 1, 1), 100)
    _plant(a, rng, TOP, 300)
    b = synth.make_b((N, K, 1, 1), 101) * np.float32(1e-30)
    _check(op, orc, a, F32, b, (M, K, 1, 1), (N, K, 1, 1), f"top binade in a, N={N}")


@pytest.mark.parametrize("N", [100, 24])
def test_top_binade_in_src1(op, orc, N):
    """b (the gradient) holds values at and next to FLT_MAX, a ~ 1e-30."""
    rng = np.random.default_rng(2)
    M, K = 160, 72
    a = synth.make_a(F32, (M, K, 1, 1), 102) * np.float32(1e-30)
    b = synth.make_b((N, K, 1, 1), 103)
    _plant(b, rng, TOP, 120)
    _check(op, orc, a, F32, b, (M, K, 1, 1), (N, K, 1, 1), f"top binade in b, N={N}")


@pytest.mark.parametrize("tid", [Q8, Q4])
def test_top_binade_gradient_quantised_src0(op, orc, tid):
    """A quantised weight against a gradient holding FLT_MAX-sized entries:
    the gradient's split must stay finite; weight scales of 6e-8 .. 1.2e-7
    keep every product finite."""
    rng = np.random.default_rng(3)
    M, K, N = 128, 64, 96
    a = _blocks(tid, rng, M, K, [0x0001, 0x0002, 0x8001])     # |d| ~ 6e-8 .. 1.2e-7
    b = synth.make_b((N, K, 1, 1), 104) * np.float32(1e-31)
    _plant(b, rng, TOP, 60)
    _check(op, orc, a, tid, b, (M, K, 1, 1), (N, K, 1, 1), f"top binade gradient, type {tid}")


@pytest.mark.parametrize("scale", [1e-20, 3e-20, 1e-19])
@pytest.mark.parametrize("N", [100, 24])
def test_subnormal_products(op, orc, scale, N):
    """a, b ~ `scale`: every product (~1e-40 .. 1e-38) is at or below fp32's
    smallest normal, and so are most sums.  No product is flushed to zero;
    each is within half a subnormal spacing (2^-150) of exact, as fp32 itself
    allows, on top of the relative bound."""
    M, K = 160, 72
    a = synth.make_a(F32, (M, K, 1, 1), 105) * np.float32(scale)
    b = synth.make_b((N, K, 1, 1), 106) * np.float32(scale)
    _check(op, orc, a, F32, b, (M, K, 1, 1), (N, K, 1, 1), f"subnormal products {scale}",
           terms=K)


def _blocks(tid, rng, M, K, scales):
    """K rows of M/32 hand-made blocks: every scale from `scales` (binary16
    bit patterns), codes uniform over the whole code range."""
    nb = M // 32
    size = 34 if tid == Q8 else 18
    out = np.zeros((1, 1, K, nb * size), dtype=np.uint8)
    blk = out.reshape(K * nb, size)
    d = np.asarray(scales, dtype=np.uint16)[rng.integers(0, len(scales), K * nb)]
    blk[:, 0] = d & 0xFF
    blk[:, 1] = d >> 8
    blk[:, 2:] = rng.integers(0, 256, (K * nb, size - 2), dtype=np.uint8)
    return out


@pytest.mark.parametrize("tid", [Q8, Q4])
def test_extreme_block_scales_bit_exact(op, orc, tid):
    """b = identity: dst reproduces the dequantised weight bit for bit with
    scales at binary16's extremes (smallest subnormal 0x0001, largest
    subnormal 0x03FF, largest finite 0x7BFF and its negative, -0 0x8000) and
    every code, including -128 for q8_0."""
    rng = np.random.default_rng(5)
    M, K = 256, 40
    a = _blocks(tid, rng, M, K, [0x0001, 0x03FF, 0x7BFF, 0xFBFF, 0x8000, 0x3C00])
    b = np.eye(K, dtype=np.float32).reshape(1, 1, K, K)
    rows = a.reshape(K, -1)
    deq = np.stack([orc.dequant_row(tid, rows[k], M) for k in range(K)])
    for p in (op.PATH_AUTO, op.PATH_TCGEN05, op.PATH_SIMT):
        got = _run(op, a, tid, b, (M, K, 1, 1), p)[0, 0].astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, deq), f"path {p}: {np.count_nonzero(got != deq)} differ"


@pytest.mark.parametrize("tid", [Q8, Q4])
def test_extreme_block_scales_outlier_gradient(op, orc, tid):
    """The same extreme scales against a gradient with 1.5e5 outliers:
    |products| up to 65504 * 128 * 1.5e5 ~ 1.3e12, all finite."""
    rng = np.random.default_rng(6)
    M, K, N = 256, 300, 100
    a = _blocks(tid, rng, M, K, [0x0001, 0x03FF, 0x7BFF, 0xFBFF, 0x8000, 0x3C00])
    b = synth.make_b((N, K, 1, 1), 112, std=1e3, outliers=True)
    _check(op, orc, a, tid, b, (M, K, 1, 1), (N, K, 1, 1), f"extreme scales, type {tid}")


@pytest.mark.parametrize("case", ["top", "subnormal"])
def test_mul_mat_id_back_range(op, orc, case):
    """MUL_MAT_ID_BACK (f32 W) at fp32's extremes, on both kernels."""
    import torch
    rng = np.random.default_rng(7)
    K, N, E, n_used, T = 192, 80, 4, 2, 40
    W = synth.normal(synth.tensor_seed(113), K * N * E).reshape(E, N, K)
    g = synth.normal(synth.tensor_seed(114), N * n_used * T).reshape(T, n_used, N)
    if case == "top":
        _plant(W, rng, TOP, 200)
        g = g * np.float32(1e-30)
    else:
        W = W * np.float32(2e-20)
        g = g * np.float32(2e-20)
    ids = synth.routing_ids(synth.tensor_seed(115), E, n_used, T)
    ref = orc.mul_mat_id_back(W, F32, ids, g, (K, N, E))
    tW, tids, tg = (torch.from_numpy(x).cuda() for x in (W, ids, g))
    for p in (op.PATH_TCGEN05, op.PATH_SIMT):
        out = op.mul_mat_id_back(tW, tids, tg, path=p)
        torch.cuda.synchronize()
        assert op.device_status() == 0
        assert_parity(out.cpu().numpy(), ref["f64"], ref["abs"], f"mmid {case} path {p}",
                      terms=N)
