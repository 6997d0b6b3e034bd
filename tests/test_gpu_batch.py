"""GPU parity of the batched narrow OUT_PROD and of the LoRA backward call,
against the CPU oracle, through the C ABI.

The rank-r gradients of LoRA fine-tuning ("metal: OUT_PROD runs batched,
broadcast and narrow shapes on the GPU", opening list item 2 and its Measured
paragraph: rank 4 / 8 / 24 gradients at the 4B's shapes) are many small
OUT_PRODs; a batch streams them through one persistent launch.
"""

import numpy as np
import pytest

import synth
from helpers import assert_parity

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


def _problem(seed, M, K, N):
    a = synth.make_a(F32, (M, K, 1, 1), seed)[0, 0]                    # (K, M)
    b = synth.make_b((N, K, 1, 1), seed + 1, std=100.0, outliers=True)[0, 0]   # (K, N)
    return a, b


def _oracle(orc, a, b):
    K, M = a.shape
    N = b.shape[1]
    r = orc.out_prod(a.reshape(1, 1, K, M), F32, b.reshape(1, 1, K, N), (M, K, 1, 1),
                     (N, K, 1, 1))
    return r["f64"][0, 0], r["abs"][0, 0]                              # (N, M)


@pytest.mark.parametrize("N", [4, 8, 24, 32])
def test_batch_mixed_list(op, orc, N):
    """Problems of different M (ragged m-tiles) and K (ragged k-stages), one
    with a transposed dst, one with M % 4 != 0 (its own launch), one with
    K == 0 (zeros), all in one call."""
    import torch
    shapes = [(2560, 512, False), (1024, 300, True), (4096, 77, False), (130, 512, False),
              (96, 0, False), (9728, 512, True), (260, 64, False)]
    probs, refs = [], []
    for i, (M, K, tr) in enumerate(shapes):
        a, b = _problem(200 + 3 * i, M, K, N)
        ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
        dst = torch.full((M, N) if tr else (N, M), float("nan"), device="cuda")
        probs.append((ta, tb, dst, tr))
        refs.append(_oracle(orc, a, b) if K else (np.zeros((N, M)), np.zeros((N, M))))
    op.out_prod_batch(probs)
    torch.cuda.synchronize()
    assert op.device_status() == 0
    for (ta, tb, dst, tr), (f64, ab), (M, K, _) in zip(probs, refs, shapes):
        got = dst.cpu().numpy()
        if tr:
            got = got.T
        assert_parity(got, f64, ab, f"batch N={N} M={M} K={K} transposed={tr}")


def test_batch_launches_and_many_problems(op, orc):
    """More problems than one launch holds: several launches, every result
    right; eligible problems share launches."""
    import torch
    n_max = op.lib().oop_out_prod_batch_max()
    count = n_max + 5
    probs, refs = [], []
    for i in range(count):
        M, K = 128 * (1 + i % 3), 64 + 32 * (i % 4)
        a, b = _problem(300 + 2 * i, M, K, 8)
        probs.append((torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                      torch.empty((8, M), device="cuda")))
        refs.append(_oracle(orc, a, b))
    op.out_prod_batch(probs)
    assert op.last_launch_count() == 2
    torch.cuda.synchronize()
    for (_, _, dst), (f64, ab) in zip(probs, refs):
        assert_parity(dst.cpu().numpy(), f64, ab, "many problems")


@pytest.mark.parametrize("r", [4, 8, 24])
def test_lora_backward_one_projection(op, orc, r):
    """The q projection of the 4B (K_in 2560 -> N_out 4096) at rank r over 512
    tokens: dA = OUT_PROD(x, dh) {2560, r}, dB = OUT_PROD(h, dz) {r, 4096},
    in one launch."""
    import torch
    K_in, N_out, T = 2560, 4096, 512
    x = synth.make_a(F32, (K_in, T, 1, 1), 320)[0, 0]                  # (T, K_in)
    dz = synth.make_b((N_out, T, 1, 1), 321, std=100.0, outliers=True)[0, 0]   # (T, N_out)
    h = synth.make_b((r, T, 1, 1), 322)[0, 0]                          # (T, r)
    dh = synth.make_b((r, T, 1, 1), 323, std=100.0, outliers=True)[0, 0]
    tx, tdz, th, tdh = (torch.from_numpy(v).cuda() for v in (x, dz, h, dh))
    dA, dB = op.lora_backward(tx, th, tdz, tdh)
    assert op.last_launch_count() == 1
    torch.cuda.synchronize()
    refA = orc.out_prod(x.reshape(1, 1, T, K_in), F32, dh.reshape(1, 1, T, r), (K_in, T, 1, 1),
                        (r, T, 1, 1))
    refB = orc.out_prod(h.reshape(1, 1, T, r), F32, dz.reshape(1, 1, T, N_out), (r, T, 1, 1),
                        (N_out, T, 1, 1))
    assert_parity(dA.cpu().numpy(), refA["f64"][0, 0], refA["abs"][0, 0], "dA")
    assert_parity(dB.cpu().numpy(), refB["f64"][0, 0], refB["abs"][0, 0], "dB")


def test_batch_rejects_before_enqueueing(op):
    """A transposed dst with N % 4 != 0 is refused before anything runs."""
    import torch
    a = torch.ones((64, 128), device="cuda")
    b = torch.ones((64, 6), device="cuda")
    d0 = torch.full((6, 128), 7.0, device="cuda")
    d1 = torch.full((128, 6), 7.0, device="cuda")
    with pytest.raises(op.OopError) as e:
        op.out_prod_batch([(a, b, d0), (a, b, d1, True)])
    assert e.value.status == op.ERR_SHAPE
    torch.cuda.synchronize()
    assert bool((d0 == 7.0).all()) and bool((d1 == 7.0).all())
