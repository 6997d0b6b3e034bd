"""Shared helpers for the GPU parity tests (no arithmetic of the method)."""

import numpy as np

TOL = 2e-6          # |gpu - exact| <= TOL * sum_k |a*b| per element


def gate(gpu, exact_f64, abssum):
    """Boolean mask of elements inside the acceptance bound."""
    g = np.asarray(gpu, dtype=np.float64)
    return np.abs(g - exact_f64) <= TOL * abssum


def assert_parity(gpu, exact_f64, abssum, what=""):
    g = np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{what}: {np.count_nonzero(~np.isfinite(g))} non-finite outputs"
    ok = gate(g, exact_f64, abssum)
    if not np.all(ok):
        err = np.abs(g.astype(np.float64) - exact_f64)
        ratio = err / np.maximum(TOL * abssum, 1e-300)
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(
            f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside 2e-6*sum|ab|; worst at {i}: "
            f"gpu={g[i]!r} exact={exact_f64[i]!r} abssum={abssum[i]!r} ratio={ratio[i]:.3g}")
    return float(np.max(np.abs(g.astype(np.float64) - exact_f64) /
                        np.maximum(TOL * abssum, 1e-300))) if g.size else 0.0


def sample_coords(rng, dims, count):
    """Random coordinates inside ``dims`` plus every corner."""
    dims = list(dims)
    pts = [rng.integers(0, d, count) for d in dims]
    c = np.stack(pts, 1)
    corners = np.array(np.meshgrid(*[[0, d - 1] for d in dims], indexing="ij")).reshape(len(dims), -1).T
    return np.concatenate([c, corners], 0).astype(np.int64)
