"""Shared helpers for the GPU parity tests (no arithmetic of the method)."""

import numpy as np

TOL = 2e-6          # |gpu - exact| <= TOL * sum_k |a*b| per element
# fp32 has no value between multiples of 2^-149 below 2^-126: an fp32 result
# cannot lie closer to the exact sum than half that spacing, and every fp32
# product a*b that falls there is itself rounded to a multiple of it.  So the
# relative bound is taken on top of an absolute floor of (terms + 1) * 2^-150:
# half a spacing for each of the `terms` products and one for the output.  For
# a result in the normal range this floor is far inside the relative bound;
# only sums of products near or below 2^-126 feel it.
FP32_HALF_SPACING = 2.0 ** -150


def _allow(abssum, terms):
    return TOL * abssum + (terms + 1) * FP32_HALF_SPACING


def gate(gpu, exact_f64, abssum, terms=0):
    """Boolean mask of elements inside the acceptance bound (`terms`: the
    number of products in each sum, for the fp32 underflow floor)."""
    g = np.asarray(gpu, dtype=np.float64)
    return np.abs(g - exact_f64) <= _allow(abssum, terms)


def assert_parity(gpu, exact_f64, abssum, what="", terms=0):
    g = np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{what}: {np.count_nonzero(~np.isfinite(g))} non-finite outputs"
    ok = gate(g, exact_f64, abssum, terms)
    if not np.all(ok):
        err = np.abs(g.astype(np.float64) - exact_f64)
        ratio = err / np.maximum(_allow(abssum, terms), 1e-300)
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(
            f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside 2e-6*sum|ab|; worst at {i}: "
            f"gpu={g[i]!r} exact={exact_f64[i]!r} abssum={abssum[i]!r} ratio={ratio[i]:.3g}")
    return float(np.max(np.abs(g.astype(np.float64) - exact_f64) /
                        np.maximum(_allow(abssum, terms), 1e-300))) if g.size else 0.0


def sample_coords(rng, dims, count):
    """Random coordinates inside ``dims`` plus every corner."""
    dims = list(dims)
    pts = [rng.integers(0, d, count) for d in dims]
    c = np.stack(pts, 1)
    corners = np.array(np.meshgrid(*[[0, d - 1] for d in dims], indexing="ij")).reshape(len(dims), -1).T
    return np.concatenate([c, corners], 0).astype(np.int64)
