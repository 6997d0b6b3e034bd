"""GPU parity of OUT_PROD for every src0 type against the CPU oracle.

OUT_PROD is instantiated for f32, f16, bf16, q4_0, q4_1, q5_0, q5_1, q8_0 and
q2_K .. q6_K ("Metal kernel_mul_mat_id_back", first bullet: out_prod's set);
the dense timings of "metal: OUT_PROD multiplies in float staging" (answer
(2)) use a q4_K weight.  Every case checks, element by element,
|gpu - exact| <= 2e-6 * sum_k |a*b| and zero non-finite outputs, on the
tensor-core kernel (TMA-fed when src0's rows are 16-byte aligned, direct loads
otherwise) and the CUDA-core kernel.
"""

import numpy as np
import pytest

import synth
from helpers import assert_parity, sample_coords

pytestmark = pytest.mark.gpu

ALL = (synth.TYPE_F16, synth.TYPE_BF16) + synth.QUANT_TYPES
KQ = (synth.TYPE_Q2_K, synth.TYPE_Q3_K, synth.TYPE_Q4_K, synth.TYPE_Q5_K, synth.TYPE_Q6_K)


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


def _src0(tid, ne, seed, std=0.02):
    """src0 bytes of `tid` ((ne3, ne2, ne1, row bytes) uint8, or 2-byte
    elements for f16 / bf16) from N(0, std) weights."""
    x = synth.normal(synth.tensor_seed(seed), int(np.prod(ne)), std=std)
    x = x.reshape(ne[3], ne[2], ne[1], ne[0])
    q = synth.quantize(tid, x)
    return q.view(np.int16) if tid in (synth.TYPE_F16, synth.TYPE_BF16) else q


def _run(op, a, tid, b, ne_a, path):
    import torch
    ta = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tb = torch.from_numpy(np.ascontiguousarray(b)).cuda()
    out = op.out_prod(ta, tb, a_type=tid, ne_a=ne_a, path=path)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    return out.cpu().numpy()


def _rows_aligned(tid, M):
    return synth.row_bytes(tid, M) % 16 == 0


@pytest.mark.parametrize("tid", ALL)
def test_every_type_whole_tensor(op, orc, tid):
    """Several m-, n- and k-tiles with ragged n and k tails, broadcast over
    two slices; the tensor-core kernel TMA-fed (aligned rows)."""
    qk = synth.BLOCK.get(tid, (1, 2))[0]
    M = 512 if qk == 256 else 384
    ne_a, ne_b = (M, 200, 1, 1), (130, 200, 2, 1)
    a = _src0(tid, ne_a, 170 + tid)
    b = synth.make_b(ne_b, 171, std=1e3, outliers=True)
    ref = orc.out_prod(a, tid, b, ne_a, ne_b)
    for p in (op.PATH_AUTO, op.PATH_TCGEN05, op.PATH_SIMT):
        assert_parity(_run(op, a, tid, b, ne_a, p), ref["f64"], ref["abs"], f"type {tid} path {p}")


@pytest.mark.parametrize("tid", ALL)
def test_every_type_unaligned_rows(op, orc, tid):
    """Rows whose byte length is not a multiple of 16: the tensor-core
    producer loads src0 directly instead of through TMA."""
    qk = synth.BLOCK.get(tid, (1, 2))[0]
    for M in ((256, 768) if qk == 256 else (96, 160, 200)):
        if qk == 1 and M % 8 == 0:
            M += 4                                   # 2-byte elements: not a multiple of 8
        if M % qk or _rows_aligned(tid, M):
            continue
        ne_a, ne_b = (M, 100, 1, 1), (97, 100, 1, 1)
        a = _src0(tid, ne_a, 172 + tid)
        b = synth.make_b(ne_b, 173, std=1e3, outliers=True)
        ref = orc.out_prod(a, tid, b, ne_a, ne_b)
        for p in (op.PATH_TCGEN05, op.PATH_SIMT):
            assert_parity(_run(op, a, tid, b, ne_a, p), ref["f64"], ref["abs"],
                          f"type {tid} M {M} path {p}")


# the block types whose rows can miss TMA's 16-byte rule, and the largest
# row group they can need (16 / gcd(block bytes, 16))
ROW_GROUPS = {synth.TYPE_Q4_1: 4, synth.TYPE_Q5_0: 8, synth.TYPE_Q5_1: 2, synth.TYPE_Q2_K: 4,
              synth.TYPE_Q3_K: 8, synth.TYPE_Q6_K: 8}


def _group(row_bytes):
    g = 1
    while row_bytes * g % 16:
        g *= 2
    return g


@pytest.mark.parametrize("tid", sorted(ROW_GROUPS))
def test_row_groups_stage_unaligned_rows(op, orc, tid):
    """Rows whose byte length is not a multiple of 16, with K a multiple of
    the row group: the TMA stages groups of 2, 4 or 8 rows (one box per
    member, the smallest group whose bytes are a multiple of 16) and the
    producer finds each row at its member's offset.  Every group size the
    type can need, ragged n and k tails, two slices of src1."""
    qk = synth.BLOCK[tid][0]
    seen = set()
    for blocks in range(1, 17):
        M = blocks * qk
        if M % 128 and qk == 256:
            continue
        g = _group(synth.row_bytes(tid, M))
        if g == 1 or g in seen:
            continue
        seen.add(g)
        assert ROW_GROUPS[tid] % g == 0
        K = 88
        ne_a, ne_b = (M, K, 1, 1), (150, K, 2, 1)
        a = _src0(tid, ne_a, 179 + tid + g)
        b = synth.make_b(ne_b, 180, std=1e3, outliers=True)
        ref = orc.out_prod(a, tid, b, ne_a, ne_b)
        assert_parity(_run(op, a, tid, b, ne_a, op.PATH_TCGEN05), ref["f64"], ref["abs"],
                      f"type {tid} M {M} K {K} groups of {g}")
    want = {2, 4, 8} if ROW_GROUPS[tid] == 8 else {2, 4} if ROW_GROUPS[tid] == 4 else {2}
    assert seen == want, seen


@pytest.mark.parametrize("tid", ALL)
def test_identity_gradient_reproduces_decoded_src0(op, orc, tid):
    """b = identity: the CUDA-core kernel returns the decoded src0 exactly as
    fp32 rounds the oracle's exact value (each decoder rounds once); the
    tensor-core kernel returns it bit for bit where the value splits into two
    TF32 terms exactly, and within 2^-21 where it carries 24 bits."""
    qk = synth.BLOCK.get(tid, (1, 2))[0]
    M, K = (512 if qk == 256 else 256), 40
    a = _src0(tid, (M, K, 1, 1), 174 + tid, std=0.5)
    rows = np.ascontiguousarray(a).view(np.uint8).reshape(K, -1)
    deq = np.stack([orc.dequant_row(tid, rows[k], M) for k in range(K)])
    want = deq.astype(np.float32).astype(np.float64)
    b = np.eye(K, dtype=np.float32).reshape(1, 1, K, K)
    simt = _run(op, a, tid, b, (M, K, 1, 1), op.PATH_SIMT)[0, 0].astype(np.float64)
    assert np.array_equal(simt, want), f"{np.count_nonzero(simt != want)} differ"
    tc = _run(op, a, tid, b, (M, K, 1, 1), op.PATH_TCGEN05)[0, 0].astype(np.float64)
    exact_split = tid in (synth.TYPE_F16, synth.TYPE_BF16, synth.TYPE_Q4_0, synth.TYPE_Q5_0,
                          synth.TYPE_Q8_0, synth.TYPE_Q3_K)
    if exact_split:
        assert np.array_equal(tc, want), f"{np.count_nonzero(tc != want)} differ"
    else:
        assert np.all(np.abs(tc - want) <= 2.0 ** -21 * np.abs(want))


@pytest.mark.parametrize("tid", [synth.TYPE_Q4_K, synth.TYPE_Q6_K, synth.TYPE_Q5_1])
def test_dense_shape_full_size_sampled(op, orc, tid):
    """The dense training shape m5120 k5120 n1024 with the pages' q4_K weight
    (and q6_K, q5_1): sampled elements against the oracle, zero non-finite."""
    import torch
    M, K, N = 5120, 5120, 1024
    x = synth.normal(synth.tensor_seed(30), M * K, std=0.02).reshape(1, 1, K, M)
    a = synth.quantize(tid, x)
    b = synth.make_b((N, K, 1, 1), 31, std=1e3, outliers=True)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = op.out_prod(ta, tb, a_type=tid, ne_a=(M, K, 1, 1))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(175 + tid)
    coords = sample_coords(rng, (M, N, 1, 1), 1500)
    val, ab = orc.out_prod_at(a, tid, b, (M, K, 1, 1), (N, K, 1, 1), coords)
    got = out.cpu().numpy()[coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]]
    assert_parity(got, val, ab, f"type {tid} dense full size")


@pytest.mark.parametrize("tid", [synth.TYPE_Q4_K, synth.TYPE_F16])
def test_backward_pair_with_new_weight_types(op, orc, tid):
    """dx of a MUL_MAT whose frozen weight is q4_K / f16, through the pair."""
    import torch
    ne_w, ne_x = (512, 96, 1, 1), (512, 40, 1, 1)
    W = _src0(tid, ne_w, 176)
    x = synth.make_b((512, 40, 1, 1), 177)
    dy = synth.make_b((96, 40, 1, 1), 178, std=1e3, outliers=True)
    ref = orc.mul_mat_back(W, tid, x, dy, ne_w)
    dW, dx = op.mul_mat_back(torch.from_numpy(W).cuda(), torch.from_numpy(x).cuda(),
                             torch.from_numpy(dy).cuda(), w_type=tid, ne_w=ne_w)
    torch.cuda.synchronize()
    assert_parity(dx.cpu().numpy(), ref["dx"]["f64"], ref["dx"]["abs"], "dx")
    assert_parity(dW.cpu().numpy(), ref["dW"]["f64"], ref["dW"]["abs"], "dW")


def test_quantised_m_must_fill_blocks(op):
    import torch
    a = torch.zeros((1, 1, 4, 144), dtype=torch.uint8, device="cuda")     # one q4_K block
    b = torch.zeros((1, 1, 4, 8), device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod(a, b, a_type=op.TYPE_Q4_K, ne_a=(128, 4, 1, 1))
    assert e.value.status == op.ERR_SHAPE
