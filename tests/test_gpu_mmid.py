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


def _run(op, W, wt, ids, g, path=None):
    import torch
    if wt == synth.TYPE_BF16:
        tW = torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).cuda()
    else:
        tW = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    out = op.mul_mat_id_back(tW, torch.from_numpy(ids).cuda(), torch.from_numpy(g).cuda(),
                             w_type=wt, path=op.PATH_AUTO if path is None else path)
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


def test_one_hot_matches_out_prod(op):
    """Every slot routed to one expert: MUL_MAT_ID_BACK equals OUT_PROD of
    that expert with the transposed gradient (both on the GPU)."""
    import torch
    K, N, E, n_used, T = 256, 96, 4, 2, 40
    W = synth.normal(63, K * N * E).reshape(E, N, K)
    g = synth.normal(64, N * n_used * T).reshape(T, n_used, N)
    ids = np.full((T, n_used), 2, np.int32)
    dx = _run(op, W, synth.TYPE_F32, ids, g).cpu().numpy()
    for i in range(n_used):
        bT = torch.from_numpy(np.ascontiguousarray(g[:, i, :].T)).cuda()   # (N, T)
        a = torch.from_numpy(np.ascontiguousarray(W[2])).cuda()            # (N, K)
        d = op.out_prod(a, bT, path=op.PATH_SIMT).cpu().numpy()          # (T, K)
        assert np.allclose(d, dx[:, i, :], rtol=0, atol=1e-5 * np.abs(d).max())


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
