"""CPU checks of the parity-test helpers themselves (tests/gpu_util.py): the slab-vectorised score
bound equals the per-row definition, the checker accepts scores inside the bound and rejects a
score just outside it, and the vectorised set overlap equals a plain set computation."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import check_scores, overlap, tolerance_row, tolerance_rows, window


@pytest.fixture(scope="module")
def tiny():
    return W.make_config("tiny")


def test_tolerance_rows_matches_definition(tiny):
    wl = tiny
    rows = np.array([0, 1, 17, 128, 255])
    b = tolerance_rows(wl, rows)
    for r, t in enumerate(rows):
        lo, hi = window(wl, int(t))
        np.testing.assert_allclose(b[r, lo:hi], tolerance_row(wl, int(t), lo, hi), rtol=1e-12, atol=0)


def test_check_scores_accepts_and_rejects(tiny):
    wl = tiny
    rows = np.arange(wl.T)
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows)
    dense = ref.dense(wl.N).astype(np.float32)  # NaN outside the windows, as an unwritten buffer
    assert check_scores(wl, dense, rows, ref, slab=64) <= 1.0
    # one in-window score moved by twice its bound is caught, in any slab
    t, j = 200, 150
    bad = dense.copy()
    bad[t, j] += np.float32(2 * tolerance_rows(wl, [t])[0, j])
    with pytest.raises(AssertionError):
        check_scores(wl, bad, rows, ref, slab=64)
    # a NaN inside a window is caught; one outside every window is not read
    bad = dense.copy()
    bad[t, 0] = np.nan
    with pytest.raises(AssertionError):
        check_scores(wl, bad, rows, ref, slab=64)
    ok = dense.copy()
    ok[t, t + 1] = np.nan  # key t + 1 is outside token t's causal window
    check_scores(wl, ok, rows, ref, slab=64)


def test_overlap_matches_sets():
    rng = np.random.default_rng(5)
    a = rng.integers(-1, 50, size=(40, 12))
    b = rng.integers(-1, 50, size=(40, 12))
    inter = total = 0
    for x, y in zip(a, b):
        sx, sy = {int(v) for v in x if v >= 0}, {int(v) for v in y if v >= 0}
        inter += len(sx & sy)
        total += len(sy)
    assert overlap(a, b) == pytest.approx(inter / total)
    assert overlap(b, b) == 1.0
    assert overlap(np.full((3, 4), -1), b[:3]) == 0.0
