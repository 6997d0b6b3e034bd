"""GPU parity of the tensor-core OUT_PROD under both tile schedules.

Data-parallel: one 128 (m) x 128 (n) dst tile per CTA.  Stream-K: one CTA per SM
shares the (tile, k-block) iterations, tiles split between CTAs are summed by
a fix-up kernel.  Both must meet |gpu - exact| <= 2e-6 * sum_k |a*b| against
the oracle, stream-K must repeat bit for bit, and the call must enqueue the
kernels it claims (split pass + tile kernel, + fix-up for stream-K).  The
shapes are small enough that forced stream-K gives every CTA only a few
k-blocks, so most tiles are shared by several CTAs (the fix-up's hard case).
"""

import numpy as np
import pytest

import synth
from helpers import assert_parity

pytestmark = pytest.mark.gpu

F32, Q8, Q4 = synth.TYPE_F32, synth.TYPE_Q8_0, synth.TYPE_Q4_0


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    yield g
    g.set_tc_schedule(g.SCHEDULE_AUTO)


CASES = [
    # (type, ne_a, ne_b): ragged m, n and k tails; slices with broadcast
    (Q8, (640, 1000, 1, 1), (300, 1000, 1, 1)),
    (Q4, (384, 4096, 1, 1), (256, 4096, 1, 1)),
    (F32, (200, 300, 2, 1), (70, 300, 4, 3)),
    (F32, (130, 33, 1, 1), (129, 33, 1, 1)),
]


def _run(op, ta, tb, a_type, ne_a, schedule, workspace=None):
    import torch
    op.set_tc_schedule(schedule)
    try:
        out = op.out_prod(ta, tb, a_type=a_type, ne_a=ne_a, path=op.PATH_TCGEN05,
                          workspace=workspace)
        n = op.last_launch_count()
        torch.cuda.synchronize()
    finally:
        op.set_tc_schedule(op.SCHEDULE_AUTO)
    assert op.device_status() == 0
    return out.cpu().numpy(), n


@pytest.mark.parametrize("a_type,ne_a,ne_b", CASES)
def test_schedules_match_oracle(op, orc, a_type, ne_a, ne_b):
    import torch
    a = synth.make_a(a_type, ne_a, 60, std=0.02 if a_type != F32 else 1.0)
    b = synth.make_b(ne_b, 61, std=1e3, outliers=True)
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    dp, n_dp = _run(op, ta, tb, a_type, ne_a, op.SCHEDULE_DATA_PARALLEL)
    sk, n_sk = _run(op, ta, tb, a_type, ne_a, op.SCHEDULE_STREAM_K)
    sk2, _ = _run(op, ta, tb, a_type, ne_a, op.SCHEDULE_STREAM_K)
    assert n_dp == 2 and n_sk == 3
    assert_parity(dp, ref["f64"], ref["abs"], f"data-parallel {a_type} {ne_a}")
    assert_parity(sk, ref["f64"], ref["abs"], f"stream-K {a_type} {ne_a}")
    assert np.array_equal(sk.view(np.uint32), sk2.view(np.uint32)), "stream-K not repeatable"


def test_minimum_workspace_runs_data_parallel(op, orc):
    """With only the minimum workspace, a forced stream-K call falls back to
    the data-parallel schedule (two launches) and stays correct."""
    import torch
    a_type, ne_a, ne_b = Q8, (640, 1000, 1, 1), (300, 1000, 1, 1)
    a = synth.make_a(a_type, ne_a, 62, std=0.02)
    b = synth.make_b(ne_b, 63, std=1e3, outliers=True)
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    need = op.oop_out_prod_workspace_min_size(a_type, ne_a, ne_b)
    full = op.oop_out_prod_workspace_size(a_type, ne_a, ne_b)
    assert 0 < need < full
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    got, n = _run(op, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), a_type, ne_a,
                  op.SCHEDULE_STREAM_K, workspace=ws)
    assert n == 2
    assert_parity(got, ref["f64"], ref["abs"], "minimum workspace")


def test_below_minimum_workspace_rejected(op):
    import torch
    ne_a, ne_b = (640, 1000, 1, 1), (300, 1000, 1, 1)
    need = op.oop_out_prod_workspace_min_size(Q8, ne_a, ne_b)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    ta = torch.zeros(1000 * 640 // 32 * 34, dtype=torch.uint8, device="cuda")
    tb = torch.zeros((1000, 300), dtype=torch.float32, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod(ta, tb, a_type=Q8, ne_a=ne_a, path=op.PATH_TCGEN05, workspace=ws)
    assert e.value.status == op.ERR_WORKSPACE
    assert op.last_launch_count() == 0


def test_auto_schedule_choice(op):
    """The automatic schedule takes stream-K exactly when an even share of
    the iterations, plus the fix-up launch (~8 k-blocks) and the partials of
    the split tail tiles (~6 per two of them a CTA), costs fewer k-block times
    than the data-parallel waves (tiles / SMs, rounded up, times the k-blocks
    per tile), and never when the tiles fill whole waves; shown on the dense
    shapes and on small problems: a wave that is mostly empty with long K
    (stream-K), short K (data-parallel), a single tile."""
    import torch
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 160)
    for m, k, n in ((5120, 5120, 1024), (5120, 17408, 1024), (1536, 1536, 1024),
                    (256, 8192, 96), (512, 4096, 256), (1024, 512, 128), (128, 2048, 96),
                    (1536, 1536, 256)):
        ta = torch.zeros(k * m // 32 * 34, dtype=torch.uint8, device="cuda")
        tb = torch.zeros((k, n), dtype=torch.float32, device="cuda")
        op.out_prod(ta, tb, a_type=Q8, ne_a=(m, k, 1, 1), path=op.PATH_TCGEN05)
        got = op.last_launch_count()
        torch.cuda.synchronize()
        tiles = -(-m // 128) * -(-n // 128)
        nkb = -(-k // 32)
        g = min(sms, tiles * nkb)
        dp = -(-tiles // g) * nkb
        tail = tiles % g
        sk = -(-(tiles * nkb) // g) + 8 + 6 * -(-(2 * tail) // g)
        want_sk = tail != 0 and sk < dp
        assert got == (3 if want_sk else 2), (m, k, n, got)


@pytest.mark.parametrize("wt", [synth.TYPE_F32, synth.TYPE_BF16])
def test_grouped_mul_mat_id_back_schedules(op, orc, wt):
    """MUL_MAT_ID_BACK's grouped product under its three schedules: persistent
    whole tiles round-robin (the default: routing, split, tile kernel), stream-K
    over the device-side work list (+ the fix-up) and data-parallel; all match
    the oracle and the default repeats bit for bit."""
    import torch
    K, N, E, n_used, T = 300, 136, 7, 3, 110
    W = synth.normal(70, K * N * E, std=0.02).reshape(E, N, K)
    if wt == synth.TYPE_BF16:
        W = synth.to_bf16_bits(W)
    ids = synth.routing_ids(71, E, n_used, T)
    g = synth.normal(72, N * n_used * T).reshape(T, n_used, N)
    ref = orc.mul_mat_id_back(W, wt, ids, g, (K, N, E))
    tW = torch.from_numpy(np.ascontiguousarray(W).view(np.int16) if wt == synth.TYPE_BF16
                          else np.ascontiguousarray(W)).cuda()
    tids, tg = torch.from_numpy(ids).cuda(), torch.from_numpy(g).cuda()
    outs, counts = [], []
    scheds = (op.SCHEDULE_AUTO, op.SCHEDULE_AUTO, op.SCHEDULE_STREAM_K,
              op.SCHEDULE_DATA_PARALLEL)
    for sched in scheds:
        op.set_tc_schedule(sched)
        try:
            out = op.mul_mat_id_back(tW, tids, tg, w_type=wt, path=op.PATH_TCGEN05)
            counts.append(op.last_launch_count())
            torch.cuda.synchronize()
        finally:
            op.set_tc_schedule(op.SCHEDULE_AUTO)
        assert op.device_status() == 0
        outs.append(out.cpu().numpy())
    assert counts == [3, 3, 4, 3]
    for o, what in zip(outs, ("persistent", "persistent again", "stream-K", "data-parallel")):
        assert_parity(o, ref["f64"], ref["abs"], f"grouped {wt} {what}")
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_long_k_stream_k_many_ctas_per_tile(op, orc):
    """K = 262144 (8192 k-blocks) on two tiles: the automatic choice is
    stream-K, each tile is shared by ~76 CTAs and the fix-up adds ~76
    partials per element; checked on sampled elements against the oracle."""
    import torch
    m, k, n = 256, 262144, 64
    a = synth.make_a(Q8, (m, k, 1, 1), 64, std=0.02)
    b = synth.make_b((n, k, 1, 1), 65, std=1e3, outliers=True)
    out = op.out_prod(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), a_type=Q8,
                      ne_a=(m, k, 1, 1), path=op.PATH_TCGEN05)
    launches = op.last_launch_count()
    torch.cuda.synchronize()
    assert op.device_status() == 0
    assert launches == 3                                  # split, tile kernel, fix-up
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(11)
    coords = np.stack([rng.integers(0, m, 300), rng.integers(0, n, 300),
                       np.zeros(300, np.int64), np.zeros(300, np.int64)], 1).astype(np.int64)
    val, ab = orc.out_prod_at(a, Q8, b, (m, k, 1, 1), (n, k, 1, 1), coords)
    got = out[0, 0, coords[:, 1], coords[:, 0]].cpu().numpy()
    assert_parity(got, val, ab, "long K stream-K")


@pytest.mark.parametrize("a_type,ne_a,ne_b", [
    (Q8, (32, 200, 1, 1), (40, 200, 1, 1)),      # one ragged m-tile, one ragged n-tile
    (F32, (500, 96, 1, 1), (33, 96, 1, 1)),      # the narrowest tensor-core width
    (Q4, (96, 33, 1, 1), (97, 33, 1, 1)),        # one k-block of 33: ragged k, n = 96 + 1
])
def test_small_edges_both_schedules(op, orc, a_type, ne_a, ne_b):
    import torch
    a = synth.make_a(a_type, ne_a, 66, std=0.02 if a_type != F32 else 1.0)
    b = synth.make_b(ne_b, 67, std=1e3, outliers=True)
    ref = orc.out_prod(a, a_type, b, ne_a, ne_b)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    for sched in (op.SCHEDULE_DATA_PARALLEL, op.SCHEDULE_STREAM_K):
        got, _ = _run(op, ta, tb, a_type, ne_a, sched)
        assert_parity(got, ref["f64"], ref["abs"], f"edge {a_type} {ne_a} {ne_b} sched {sched}")
