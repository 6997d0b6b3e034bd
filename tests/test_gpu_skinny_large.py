"""GPU parity of the skinny-N OUT_PROD on large problems, where the library
takes its persistent TMA-fed form (at least two m-tile x slice items per SM,
N % 4 == 0, M % 4 == 0; items of 128 m up to N = 24, of 64 m above or when
128 would be too few): ragged m-tiles, K not a multiple of the 64-row stage,
broadcast slices, both item widths, outliers in b."""

import numpy as np
import pytest

import synth
from helpers import assert_parity, sample_coords

pytestmark = pytest.mark.gpu

F32 = synth.TYPE_F32


@pytest.fixture(scope="module")
def op():
    import torch
    import ggml_out_prod_gb300 as g
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.build()
    g.lib()
    return g


@pytest.mark.parametrize("ne_a,ne_b", [
    ((1000, 300, 40, 1), (8, 300, 40, 1)),       # 8 m-tiles (last ragged) x 40 slices
    ((1000, 300, 10, 1), (4, 300, 40, 1)),       # broadcast: 4 dst slices per src0 slice
    ((1000, 130, 20, 1), (24, 130, 20, 1)),      # N = 24, 160 items of 128 m: 64-wide; K = 2 stages + 2
    ((1000, 200, 40, 1), (24, 200, 40, 1)),      # N = 24, 320 items of 128 m; K = 3 stages + 8 rows
    ((640, 96, 64, 1), (20, 96, 64, 1)),         # N = 20, 128-wide, K = 1.5 stages
    ((512, 77, 5, 2), (32, 77, 20, 4)),          # N = 32, broadcast in both dims
    ((2000, 64, 30, 1), (12, 64, 30, 1)),        # K exactly one stage
])
def test_large_skinny_matches_oracle(op, orc, ne_a, ne_b):
    import torch
    a = synth.make_a(F32, ne_a, 80)
    b = synth.make_b(ne_b, 81, std=100.0, outliers=True)
    ref = orc.out_prod(a, F32, b, ne_a, ne_b)
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda()
    out = op.out_prod(ta, tb, ne_a=ne_a, path=op.PATH_SKINNY)
    assert op.last_launch_count() == 1
    torch.cuda.synchronize()
    assert op.device_status() == 0
    got = out.cpu().numpy()
    assert_parity(got, ref["f64"], ref["abs"], f"large skinny {ne_a} {ne_b}")
    again = op.out_prod(ta, tb, ne_a=ne_a, path=op.PATH_SKINNY).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32)), "not repeatable"


def test_batched_rank8_full_size_sampled(op, orc):
    """64 rank-8 gradients a [2560, 512] (335 MB of src0) in one call."""
    import torch
    ne_a, ne_b = (2560, 512, 64, 1), (8, 512, 64, 1)
    a = synth.make_a(F32, ne_a, 82)
    b = synth.make_b(ne_b, 83, std=100.0, outliers=True)
    out = op.out_prod(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), ne_a=ne_a,
                      path=op.PATH_SKINNY)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(9)
    coords = sample_coords(rng, (2560, 8, 64, 1), 2000)
    val, ab = orc.out_prod_at(a, F32, b, ne_a, ne_b, coords)
    got = out[coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]].cpu().numpy()
    assert_parity(got, val, ab, "batched rank-8")
