"""GPU parity of OUT_PROD against the CPU oracle, through the C ABI.

Every case feeds the same seeded bytes to both sides and checks, element by
element, |gpu - exact| <= 2e-6 * sum_k |a*b| and zero non-finite outputs.
At full workload sizes the oracle computes sampled elements one by one.
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


def _paths(op, a_type, N):
    ps = [op.PATH_AUTO, op.PATH_SIMT]
    if a_type == F32 and N <= 32:
        ps.append(op.PATH_SKINNY)
    if getattr(op, "HAS_TCGEN05", False):
        ps.append(op.PATH_TCGEN05)
    return ps


def _gpu(op, a, a_type, b, ne_a, path, guard=0):
    import torch
    ta = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tb = torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).cuda()
    ne_b = op.ne_of(tb)
    shape = (ne_b[3], ne_b[2], ne_b[0], ne_a[0])
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    if guard:
        buf.view(torch.int32)[:guard] = 0x7FC0DEAD
        buf.view(torch.int32)[n + guard:] = 0x7FC0DEAD
    out = buf[guard:guard + n].view(shape)
    op.out_prod(ta, tb, a_type=a_type, ne_a=ne_a, out=out, path=path)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    if guard:
        g = buf.view(torch.int32).cpu().numpy()
        assert np.all(g[:guard] == 0x7FC0DEAD) and np.all(g[n + guard:] == 0x7FC0DEAD), \
            "guard band overwritten"
    return out.cpu().numpy()


def _check_whole(op, orc, a, a_type, b, ne_a, ne_b, paths=None, what=""):
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    worst = 0.0
    for p in paths or _paths(op, a_type, ne_b[0]):
        got = _gpu(op, a, a_type, b, ne_a, p, guard=64)
        worst = max(worst, assert_parity(got, ref["f64"], ref["abs"], f"{what} path {p}"))
    return worst


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def test_single_slice(op, orc):
    a, b = synth.single_slice()
    _check_whole(op, orc, a, F32, b, (256, 512, 1, 1), (8, 512, 1, 1), what="single slice")


@pytest.mark.parametrize("r", synth.LORA_RANKS)
def test_lora_rank(op, orc, r):
    a, b = synth.lora_rank(r)
    _check_whole(op, orc, a, F32, b, (2560, 512, 1, 1), (r, 512, 1, 1), what=f"lora r={r}")


@pytest.mark.parametrize("n_seq", [1, 2])
def test_grouped_heads(op, orc, n_seq):
    a, b = synth.grouped_heads(n_seq)
    _check_whole(op, orc, a, F32, b, (128, 512, 4, n_seq), (128, 512, 16, n_seq),
                 what=f"grouped heads x{n_seq}")


@pytest.mark.parametrize("tid", [Q8, Q4])
@pytest.mark.parametrize("m,k", [(320, 300), (96, 1000)])
def test_dense_quant_small_whole(op, orc, tid, m, k):
    """Several tiles and ragged tails in n and k, checked everywhere."""
    a = synth.make_a(tid, (m, k, 1, 1), 30, std=0.02)
    b = synth.make_b((200, k, 1, 1), 31, std=1e3, outliers=True)
    _check_whole(op, orc, a, tid, b, (m, k, 1, 1), (200, k, 1, 1), what=f"dense {tid} {m}x{k}")


@pytest.mark.parametrize("tid", [Q8, Q4])
@pytest.mark.parametrize("mk", synth.DENSE_MK)
def test_dense_quant_full_sampled(op, orc, tid, mk):
    import torch
    m, k = mk
    a, b = synth.dense_quant(tid, m, k)
    ne_a, ne_b = (m, k, 1, 1), (1024, k, 1, 1)
    rng = np.random.default_rng(m * 7 + k)
    coords = sample_coords(rng, (m, 1024, 1, 1), 1500)
    val, ab = orc.out_prod_at(a, tid, b, ne_a, ne_b, coords)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    for p in [op.PATH_AUTO] + ([op.PATH_TCGEN05] if getattr(op, "HAS_TCGEN05", False) else []):
        out = op.out_prod(ta, tb, a_type=tid, ne_a=ne_a, path=p)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out).all()), "non-finite outputs"
        got = out[coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]].cpu().numpy()
        assert_parity(got, val, ab, f"dense full {tid} {mk} path {p}")


# ---------------------------------------------------------------------------
# edge cases and pins on the GPU
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ne_a,ne_b", [
    ((1, 1, 1, 1), (1, 1, 1, 1)),
    ((37, 1, 1, 1), (33, 1, 1, 1)),
    ((130, 3, 1, 1), (1, 3, 1, 1)),
    ((131, 65, 2, 1), (31, 65, 6, 1)),      # M odd: scalar loads
    ((258, 129, 1, 2), (32, 129, 3, 4)),    # M even, not /4: 8-byte loads
    ((64, 1000, 1, 1), (17, 1000, 1, 1)),
    ((300, 70, 1, 1), (33, 70, 1, 1)),      # first N on the dense side
    ((200, 4500, 1, 1), (5, 4500, 1, 1)),   # long K: several staging passes
])
def test_edge_shapes_f32(op, orc, ne_a, ne_b):
    a = synth.make_a(F32, ne_a, 50)
    b = synth.make_b(ne_b, 51, std=100.0, outliers=ne_b[0] * ne_b[1] > 500)
    _check_whole(op, orc, a, F32, b, ne_a, ne_b, what=f"edge {ne_a} {ne_b}")


@pytest.mark.parametrize("tid,M,K,N", [(F32, 300, 1000, 130), (F32, 300, 1024, 256),
                                       (Q8, 320, 300, 200), (Q4, 288, 200, 70)])
def test_ragged_tiles_repeatable(op, orc, tid, M, K, N):
    """Ragged m-, n- and k-tiles on the tensor-core path: every repeat inside
    the bound and bit-identical to the first (the summation order is fixed)."""
    import torch
    ne_a, ne_b = (M, K, 1, 1), (N, K, 1, 1)
    a = synth.make_a(tid, ne_a, 90, std=0.02 if tid != F32 else 1.0)
    b = synth.make_b(ne_b, 91, std=1e3 if tid != F32 else 1.0, outliers=True)
    ref = orc.out_prod(a, tid, b, ne_a, ne_b)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    first = None
    for _ in range(12):
        out = op.out_prod(ta, tb, a_type=tid, ne_a=ne_a, path=op.PATH_TCGEN05).cpu().numpy()
        assert_parity(out, ref["f64"], ref["abs"], f"ragged {tid} {M}x{K}x{N}")
        if first is None:
            first = out
        else:
            assert np.array_equal(first.view(np.uint32), out.view(np.uint32)), "not repeatable"


def test_integer_inputs_exact(op, orc):
    rng = np.random.default_rng(3)
    ne_a, ne_b = (96, 77, 2, 1), (20, 77, 4, 1)
    a = rng.integers(-8, 9, size=(1, 2, 77, 96)).astype(np.float32)
    b = rng.integers(-8, 9, size=(1, 4, 77, 20)).astype(np.float32)
    ref = orc.out_prod(a, F32, b, ne_a, ne_b)
    for p in _paths(op, F32, 20):
        got = _gpu(op, a, F32, b, ne_a, p)
        assert np.array_equal(got.astype(np.float64), ref["f64"]), f"path {p}"


@pytest.mark.parametrize("tid", [F32, Q8, Q4])
def test_identity_b_reproduces_dequantised_a(op, orc, tid):
    """b = identity (N = K): dst[m, n] = a[m, n], bit for bit."""
    M, K = 256, 40
    a = synth.make_a(tid, (M, K, 1, 1), 52, std=0.5)
    b = np.eye(K, dtype=np.float32).reshape(1, 1, K, K)
    rows = a.reshape(K, -1).view(np.uint8)
    deq = np.stack([orc.dequant_row(tid, rows[k], M) for k in range(K)])
    for p in _paths(op, tid, K):
        got = _gpu(op, a, tid, b, (M, K, 1, 1), p)[0, 0].astype(np.float64)
        if tid == F32 and p in (op.PATH_TCGEN05, op.PATH_AUTO):
            # f32 src0 keeps 22 of its 24 significant bits in the TF32 pair
            assert np.all(np.abs(got - deq) <= 2.0 ** -21 * np.abs(deq)), f"path {p}"
        else:
            assert np.array_equal(got, deq), f"path {p}"


def test_broadcast_equals_replication_gpu(op):
    ne_a, ne_b = (160, 64, 2, 2), (24, 64, 6, 4)
    a = synth.make_a(F32, ne_a, 53)
    b = synth.make_b(ne_b, 54, outliers=True)
    rep = np.repeat(np.repeat(a, 3, axis=1), 2, axis=0)
    for p in _paths(op, F32, 24):
        g1 = _gpu(op, a, F32, b, ne_a, p)
        g2 = _gpu(op, rep, F32, b, (160, 64, 6, 4), p)
        assert np.array_equal(g1, g2), f"path {p}"


def test_empty_k_writes_zeros(op):
    import torch
    a = torch.empty((1, 1, 0, 64), dtype=torch.float32, device="cuda")
    b = torch.empty((1, 1, 0, 5), dtype=torch.float32, device="cuda")
    out = torch.full((1, 1, 5, 64), 7.0, device="cuda")
    op.out_prod(a, b, ne_a=(64, 0, 1, 1), out=out)
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_empty_dst_is_noop(op):
    import torch
    a = torch.ones((1, 1, 8, 64), dtype=torch.float32, device="cuda")
    b = torch.ones((1, 1, 8, 0), dtype=torch.float32, device="cuda")
    out = op.out_prod(a, b, ne_a=(64, 8, 1, 1))
    assert out.numel() == 0


def test_unaligned_src0(op, orc):
    """src0 starting 4 bytes past a 16-byte boundary takes the scalar loads."""
    import torch
    ne_a, ne_b = (128, 50, 1, 1), (8, 50, 1, 1)
    a = synth.make_a(F32, ne_a, 55)
    b = synth.make_b(ne_b, 56)
    ref = orc.out_prod(a, F32, b, ne_a, ne_b)
    buf = torch.zeros(a.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(a.reshape(-1)).cuda()
    ta = buf[1:].view(a.shape)
    for p in _paths(op, F32, 8):
        out = op.out_prod(ta, torch.from_numpy(b).cuda(), ne_a=ne_a, path=p)
        torch.cuda.synchronize()
        assert_parity(out.cpu().numpy(), ref["f64"], ref["abs"], f"unaligned path {p}")


def test_host_checks_reject(op):
    import torch
    a = torch.ones((1, 3, 8, 64), dtype=torch.float32, device="cuda")
    b = torch.ones((1, 16, 8, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod(a, b)
    assert e.value.status == op.ERR_BROADCAST
    b2 = torch.ones((1, 3, 7, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod(a, b2)
    assert e.value.status == op.ERR_SHAPE
    q = torch.zeros((1, 1, 8, 34), dtype=torch.uint8, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod(q, b[:, :3].contiguous(), a_type=op.TYPE_Q8_0, ne_a=(16, 8, 1, 1))
    assert e.value.status == op.ERR_SHAPE
    with pytest.raises(op.OopError) as e:
        op.out_prod(a, torch.ones((1, 3, 8, 40), device="cuda"), path=op.PATH_SKINNY)
    assert e.value.status == op.ERR_PATH


# ---------------------------------------------------------------------------
# the host entry (host buffers in and out, one call)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("a_type,ne_a,ne_b", [
    (Q8, (640, 1000, 1, 1), (300, 1000, 1, 1)),     # pipelined: three k chunks (224, 416, 360)
    (Q8, (256, 4096, 1, 1), (100, 4096, 1, 1)),     # long K, narrow: four k chunks
    (F32, (200, 300, 2, 1), (70, 300, 4, 3)),       # several slices: one pass
    (F32, (256, 512, 1, 1), (8, 512, 1, 1)),        # skinny-N: one pass
    (Q4, (384, 700, 1, 1), (200, 700, 1, 1)),       # two k chunks (256, 444)
    (F32, (300, 300, 1, 1), (50, 300, 1, 1)),       # K < 512: one pass
])
def test_host_entry_matches_oracle(op, orc, a_type, ne_a, ne_b):
    import torch
    a = synth.make_a(a_type, ne_a, 90, std=0.02 if a_type != F32 else 1.0)
    b = synth.make_b(ne_b, 91, std=1e3, outliers=True)
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    out = op.out_prod_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(),
                           a_type=a_type, ne_a=ne_a)
    assert op.device_status() == 0
    assert_parity(out.numpy(), ref["f64"], ref["abs"], f"host entry {a_type} {ne_a}")


def test_host_entry_rejects(op):
    import torch
    ne_a, ne_b = (640, 1000, 1, 1), (300, 1000, 1, 1)
    need = op.oop_out_prod_host_buffer_size(Q8, ne_a, ne_b)
    assert need > 0
    a = torch.zeros(1000 * 640 // 32 * 34, dtype=torch.uint8)
    b = torch.zeros((1000, 300), dtype=torch.float32)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod_host(a, b, a_type=Q8, ne_a=ne_a, device_buffer=small)
    assert e.value.status == op.ERR_WORKSPACE
    with pytest.raises(op.OopError) as e:                # K mismatch
        op.out_prod_host(a, torch.zeros((999, 300), dtype=torch.float32), a_type=Q8, ne_a=ne_a)
    assert e.value.status == op.ERR_SHAPE
