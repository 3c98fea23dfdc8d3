"""Helpers shared by the GPU parity tests: device copies, the score tolerance, comparisons.

The tolerance is the fp32 accumulation bound, in score units,
    B(t, j) = 1e-4 * |k_scale[j]| * sum_h |w[t, h]| * sum_d |q[t, h, d] k[j, d]| + 1e-6,
computed here in float64 from decoded inputs (torch's float8_e4m3fn decoder, independent of the
oracle and of the library).
"""
from __future__ import annotations

import numpy as np

import oracle as O


def decode(codes: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def to_dev(wl, device="cuda"):
    import torch

    return {name: torch.from_numpy(np.ascontiguousarray(getattr(wl, name))).to(device)
            for name in ("q", "w", "k", "k_scale", "ks", "ke")}


def window(wl, t):
    lo = min(max(int(wl.ks[t]), 0), wl.N)
    hi = min(max(int(wl.ke[t]), 0), wl.N)
    return lo, max(lo, hi)


def tolerance_row(wl, t, lo, hi, qdec=None, kdec=None):
    qv = decode(wl.q[t]) if qdec is None else qdec[t]
    kv = decode(wl.k[lo:hi]) if kdec is None else kdec[lo:hi]
    abs_dots = np.abs(kv) @ np.abs(qv).T  # [n, H]: sum_d |q k|
    return 1e-4 * np.abs(wl.k_scale[lo:hi].astype(np.float64)) * (abs_dots @ np.abs(wl.w[t].astype(np.float64))) \
        + 1e-6


def check_scores(wl, logits_rows: np.ndarray, rows, ref: O.RowScores, exact=False):
    """Every in-window GPU score of the listed rows within tolerance of the oracle (or equal).

    logits_rows[r] is the GPU logits row of token rows[r].  Returns the worst error / bound.
    """
    worst = 0.0
    kdec = decode(wl.k)
    for r, t in enumerate(rows):
        lo, n = int(ref.lo[r]), int(ref.length[r])
        if n == 0:
            continue
        g = logits_rows[r, lo:lo + n].astype(np.float64)
        o = ref.row(r)
        assert not np.any(np.isnan(g)), f"row {t}: NaN in window"
        if exact:
            bad = np.nonzero(g != o)[0]
            assert bad.size == 0, f"row {t}: {bad.size} inexact, first key {lo + bad[0]}: {g[bad[0]]} vs {o[bad[0]]}"
        else:
            b = tolerance_row(wl, t, lo, lo + n, kdec=kdec)
            ratio = np.abs(g - o) / b
            k_bad = int(np.argmax(ratio))
            assert ratio[k_bad] <= 1.0, f"row {t} key {lo + k_bad}: |{g[k_bad]} - {o[k_bad]}| > {b[k_bad]}"
            worst = max(worst, float(ratio.max()))
    return worst


def overlap(idx_a: np.ndarray, idx_b: np.ndarray) -> float:
    """sum_rows |A & B| / sum_rows |B| over valid (non -1) entries."""
    inter = 0
    total = 0
    for a, b in zip(idx_a, idx_b):
        sa = set(int(x) for x in a if x >= 0)
        sb = set(int(x) for x in b if x >= 0)
        inter += len(sa & sb)
        total += len(sb)
    return 1.0 if total == 0 else inter / total
