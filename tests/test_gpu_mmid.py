"""GPU parity of MUL_MAT_ID_BACK against the CPU oracle, through the C ABI."""

import numpy as np
import pytest

import synth
from helpers import assert_parity, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


def _run(op, W, wt, ids, g, path=None, K=None):
    import torch
    if wt in (synth.TYPE_BF16, synth.TYPE_F16):
        tW = torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).cuda()
    else:
        tW = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    out = op.mul_mat_id_back(tW, torch.from_numpy(ids).cuda(), torch.from_numpy(g).cuda(),
                             w_type=wt, path=op.PATH_AUTO if path is None else path, K=K)
    torch.cuda.synchronize()
    return out


PATHS = ["tcgen05", "simt"]


def _path(op, name):
    return op.PATH_TCGEN05 if name == "tcgen05" else op.PATH_SIMT


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wt", [synth.TYPE_F32, synth.TYPE_BF16])
def test_small_whole(op, orc, wt, path):
    K, N, E, n_used, T = 300, 136, 7, 3, 110
    W = synth.normal(60, K * N * E, std=0.02).reshape(E, N, K)
    if wt == synth.TYPE_BF16:
        W = synth.to_bf16_bits(W)
    ids = synth.routing_ids(61, E, n_used, T)
    g = synth.normal(62, N * n_used * T).reshape(T, n_used, N)
    ref = orc.mul_mat_id_back(W, wt, ids, g, (K, N, E))
    got = _run(op, W, wt, ids, g, _path(op, path)).cpu().numpy()
    assert op.device_status() == 0
    assert_parity(got, ref["f64"], ref["abs"], f"mmid small {wt} {path}")


@pytest.mark.parametrize("sched", ["auto", "stream_k"])
def test_rows_off_16_bytes(op, orc, sched):
    """dx rows of 302 floats: a row start is not always 16-byte aligned, so
    the tile kernel stores the results itself instead of copying them out in
    bulk; the stream-K schedule's shared tiles go through partial sums."""
    K, N, E, n_used, T = 302, 72, 5, 2, 90
    W = synth.normal(63, K * N * E, std=0.02).reshape(E, N, K)
    ids = synth.routing_ids(64, E, n_used, T)
    g = synth.normal(65, N * n_used * T).reshape(T, n_used, N)
    ref = orc.mul_mat_id_back(W, synth.TYPE_F32, ids, g, (K, N, E))
    op.set_tc_schedule(op.SCHEDULE_AUTO if sched == "auto" else op.SCHEDULE_STREAM_K)
    try:
        got = _run(op, W, synth.TYPE_F32, ids, g, op.PATH_TCGEN05).cpu().numpy()
    finally:
        op.set_tc_schedule(op.SCHEDULE_AUTO)
    assert op.device_status() == 0
    assert_parity(got, ref["f64"], ref["abs"], f"mmid rows off 16 bytes {sched}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wt", [synth.TYPE_F32, synth.TYPE_BF16])
def test_moe_full_sampled(op, orc, wt, path):
    import torch
    W, ids, g = synth.moe_back(wt)
    ne_w = (2048, 768, 32)
    out = _run(op, W, wt, ids, g, _path(op, path))
    assert op.device_status() == 0
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(5)
    coords = sample_coords(rng, (2048, 8, 512), 3000)
    val, ab = orc.mul_mat_id_back_at(W, wt, ids, g, ne_w, coords)
    got = out[coords[:, 2], coords[:, 1], coords[:, 0]].cpu().numpy()
    assert_parity(got, val, ab, f"mmid full {wt} {path}")


def test_skewed_routing_and_duplicates(op, orc):
    """Every token sends most slots to one expert (several n-tiles for it),
    including the same expert twice: each slot is still its own column."""
    import torch
    K, N, E, n_used, T = 256, 200, 5, 4, 300
    W = synth.normal(67, K * N * E, std=0.02).reshape(E, N, K)
    g = synth.normal(68, N * n_used * T).reshape(T, n_used, N)
    ids = np.zeros((T, n_used), np.int32)
    ids[:, 1] = 3
    ids[:, 2] = (np.arange(T) % 5).astype(np.int32)
    ids[:, 3] = 0                                             # duplicate of slot 0
    ref = orc.mul_mat_id_back(W, synth.TYPE_F32, ids, g, (K, N, E))
    for path in PATHS:
        got = _run(op, W, synth.TYPE_F32, ids, g, _path(op, path)).cpu().numpy()
        assert op.device_status() == 0
        assert_parity(got, ref["f64"], ref["abs"], f"skewed {path}")


def test_one_hot_matches_oracle_out_prod(op, orc):
    """Every slot routed to one expert: MUL_MAT_ID_BACK on the GPU equals the
    oracle's OUT_PROD of that expert with the transposed gradient, within the
    bound, on both kernels."""
    K, N, E, n_used, T = 256, 96, 4, 2, 40
    W = synth.normal(63, K * N * E).reshape(E, N, K)
    g = synth.normal(64, N * n_used * T).reshape(T, n_used, N)
    ids = np.full((T, n_used), 2, np.int32)
    for path in PATHS:
        dx = _run(op, W, synth.TYPE_F32, ids, g, _path(op, path)).cpu().numpy()
        for i in range(n_used):
            bT = np.ascontiguousarray(g[:, i, :].T).reshape(1, 1, N, T)     # b[n=t, k=r]
            ref = orc.out_prod(W[2].reshape(1, 1, N, K), synth.TYPE_F32, bT, (K, N, 1, 1),
                               (T, N, 1, 1))
            assert_parity(dx[:, i, :], ref["f64"][0, 0], ref["abs"][0, 0], f"one-hot {path}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wt", [synth.TYPE_F16, synth.TYPE_Q4_0, synth.TYPE_Q4_1, synth.TYPE_Q5_0,
                                synth.TYPE_Q5_1, synth.TYPE_Q8_0, synth.TYPE_Q2_K, synth.TYPE_Q3_K,
                                synth.TYPE_Q4_K, synth.TYPE_Q5_K, synth.TYPE_Q6_K])
def test_every_expert_type(op, orc, wt, path):
    """Expert weights of every type of "Metal kernel_mul_mat_id_back" (first
    bullet), whole tensor, ragged n-tiles, both kernels."""
    qk = synth.BLOCK.get(wt, (1, 2))[0]
    K, N, E, n_used, T = (512 if qk == 256 else 320), 136, 5, 3, 70
    x = synth.normal(69, K * N * E, std=0.02).reshape(E, N, K)
    W = synth.quantize(wt, x).reshape(E, N, -1)
    ids = synth.routing_ids(70, E, n_used, T)
    g = synth.normal(71, N * n_used * T).reshape(T, n_used, N)
    ref = orc.mul_mat_id_back(W, wt, ids, g, (K, N, E))
    got = _run(op, W, wt, ids, g, _path(op, path), K=K).cpu().numpy()
    assert op.device_status() == 0
    assert_parity(got, ref["f64"], ref["abs"], f"mmid type {wt} {path}")


@pytest.mark.parametrize("wt", [synth.TYPE_Q8_0, synth.TYPE_Q4_K])
def test_moe_full_sampled_quantised(op, orc, wt):
    """The MoE workload (E = 32 experts [2048, 768], 8 of 32 per token, 512
    tokens) with quantised expert weights, sampled against the oracle."""
    import torch
    W, ids, g = synth.moe_back(synth.TYPE_F32)
    Wq = synth.quantize(wt, W).reshape(32, 768, -1)
    out = _run(op, Wq, wt, ids, g, op.PATH_TCGEN05, K=2048)
    assert op.device_status() == 0
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(6)
    coords = sample_coords(rng, (2048, 8, 512), 3000)
    val, ab = orc.mul_mat_id_back_at(Wq, wt, ids, g, (2048, 768, 32), coords)
    got = out[coords[:, 2], coords[:, 1], coords[:, 0]].cpu().numpy()
    assert_parity(got, val, ab, f"mmid full {wt}")


@pytest.mark.parametrize("path", PATHS)
def test_bad_id_zeroes_slot_and_reports(op, path):
    import torch
    K, N, E = 64, 32, 4
    W = synth.normal(65, K * N * E).reshape(E, N, K)
    g = synth.normal(66, N * 2 * 3).reshape(3, 2, N)
    ids = np.array([[0, 1], [2, 9], [3, -1]], np.int32)
    op.device_status(clear=True)
    out = _run(op, W, synth.TYPE_F32, ids, g, _path(op, path)).cpu().numpy()
    assert op.device_status(clear=True) == op.ERR_BAD_ID
    assert np.all(out[1, 1] == 0) and np.all(out[2, 1] == 0)
    assert np.any(out[0, 0] != 0)
    assert op.device_status() == 0


# ---------------------------------------------------------------------------
# MUL_MAT_ID's expert-weight gradient
# ---------------------------------------------------------------------------

def _wgrad_inputs(seed, K, N, E, n_used, n_x, T, outliers=True):
    x = synth.normal(synth.tensor_seed(seed), T * n_x * K).reshape(T, n_x, K)
    dy = synth.make_b((N, n_used, T, 1), seed + 1, std=1e3, outliers=outliers)[0]
    ids = synth.routing_ids(synth.tensor_seed(seed + 2), E, n_used, T)
    return x, ids, dy


def _wgrad(op, x, ids, dy, E):
    import torch
    out = op.mul_mat_id_weight_grad(torch.from_numpy(x).cuda(), torch.from_numpy(ids).cuda(),
                                    torch.from_numpy(dy).cuda(), E)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("K,N,E,n_used,n_x,T", [
    (256, 96, 6, 3, 3, 70),      # one x row per slot, ragged segments
    (300, 136, 5, 4, 1, 33),     # one x row per token, ragged m and n tiles
    (128, 50, 40, 2, 2, 9),      # most experts with no slot: their gradient is zero
    (302, 72, 3, 2, 2, 20),      # dW rows of 302 floats: stored directly, not in bulk
])
def test_expert_weight_grad_whole(op, orc, K, N, E, n_used, n_x, T):
    """Both schedules: persistent (the default) and one CTA per tile."""
    x, ids, dy = _wgrad_inputs(190 + E, K, N, E, n_used, n_x, T)
    ref = orc.mul_mat_id_weight_grad(x, ids, dy, E)
    for sched in (op.SCHEDULE_AUTO, op.SCHEDULE_DATA_PARALLEL):
        op.set_tc_schedule(sched)
        try:
            got = _wgrad(op, x, ids, dy, E).cpu().numpy()
        finally:
            op.set_tc_schedule(op.SCHEDULE_AUTO)
        assert op.device_status() == 0
        assert_parity(got, ref["f64"], ref["abs"], f"expert weight grad {K}x{N}x{E} {sched}")


def test_expert_weight_grad_repeatable(op, orc):
    """The routing lays each expert's slots out in slot order, so every sum
    over an expert's slots runs in one order: repeated calls give the same
    bits.  2400 slots (three routing batches), ~300 slots an expert."""
    K, N, E, n_used, n_x, T = 256, 96, 8, 4, 2, 600
    x, ids, dy = _wgrad_inputs(198, K, N, E, n_used, n_x, T)
    first = _wgrad(op, x, ids, dy, E).cpu().numpy()
    assert op.device_status() == 0
    for _ in range(3):
        again = _wgrad(op, x, ids, dy, E).cpu().numpy()
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))
    ref = orc.mul_mat_id_weight_grad(x, ids, dy, E)
    assert_parity(first, ref["f64"], ref["abs"], "expert weight grad repeatable")


def test_expert_weight_grad_skewed(op, orc):
    """Most slots routed to one expert (a segment of many k-blocks next to
    segments of one)."""
    K, N, E, n_used, T = 192, 100, 4, 3, 200
    x, _, dy = _wgrad_inputs(195, K, N, E, n_used, n_used, T)
    ids = np.zeros((T, n_used), np.int32)
    ids[:, 1] = 2
    ids[::7, 2] = 3
    ids[1::7, 2] = 1
    ref = orc.mul_mat_id_weight_grad(x, ids, dy, E)
    got = _wgrad(op, x, ids, dy, E).cpu().numpy()
    assert_parity(got, ref["f64"], ref["abs"], "skewed")


def test_expert_weight_grad_moe_full_sampled(op, orc):
    """The MoE workload's shapes (32 experts [2048, 768], 8 of 32 per token,
    512 tokens, one x row per slot), sampled against the oracle."""
    import torch
    K, N, E, n_used, T = 2048, 768, 32, 8, 512
    x, ids, dy = _wgrad_inputs(196, K, N, E, n_used, n_used, T, outliers=False)
    out = _wgrad(op, x, ids, dy, E)
    assert op.device_status() == 0
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(197)
    got = out.cpu().numpy()
    for e in rng.choice(E, 4, replace=False):
        # expert e's gradient is the oracle's OUT_PROD over its slots in
        # slot order (t, then i), the same sums in the same order
        t_idx, i_idx = np.nonzero(ids == e)
        xs = np.ascontiguousarray(x[t_idx, i_idx % n_used])          # (cnt, K)
        ds = np.ascontiguousarray(dy[t_idx, i_idx])                  # (cnt, N)
        cnt = len(t_idx)
        ref = orc.out_prod(xs.reshape(1, 1, cnt, K), synth.TYPE_F32, ds.reshape(1, 1, cnt, N),
                           (K, cnt, 1, 1), (N, cnt, 1, 1))
        assert_parity(got[e], ref["f64"][0, 0], ref["abs"][0, 0], f"moe weight grad, expert {e}")


def test_expert_weight_grad_bad_id(op, orc):
    K, N, E = 64, 40, 3
    x, ids, dy = _wgrad_inputs(198, K, N, E, 2, 2, 5)
    ids = ids.copy()
    ids[2, 1] = 7
    op.device_status(clear=True)
    got = _wgrad(op, x, ids, dy, E).cpu().numpy()
    assert op.device_status(clear=True) == op.ERR_BAD_ID
    keep = ids.copy()
    keep[2, 1] = 0
    dy2 = dy.copy()
    dy2[2, 1] = 0                                    # that slot contributes nothing
    ref = orc.mul_mat_id_weight_grad(x, keep, dy2, E)
    assert_parity(got, ref["f64"], ref["abs"], "bad id ignored")
