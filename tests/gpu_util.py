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


def windowed_scores(dsa, t, wl, rows, slab=16):
    """GPU scores of the listed rows' windows (one array per row), scored through dsa_index_score
    in slabs of rows so that no [T, N] buffer is needed."""
    import torch

    out = []
    for s0 in range(0, len(rows), slab):
        r = torch.from_numpy(np.asarray(rows[s0:s0 + slab], dtype=np.int64)).cuda()
        sub = torch.full((len(r), wl.N), float("nan"), dtype=torch.float32, device="cuda")
        dsa.index_score(t["q"][r].contiguous(), t["w"][r].contiguous(), t["k"], t["k_scale"],
                        t["ks"][r].contiguous(), t["ke"][r].contiguous(), logits=sub)
        assert dsa.get_device_error() == 0
        for i, row in enumerate(rows[s0:s0 + slab]):
            lo, hi = window(wl, int(row))
            out.append(sub[i, lo:hi].cpu().numpy())
        del sub
    return out


def check_windowed(wl, rows, gpu_rows, ref: O.RowScores, idx_rows: np.ndarray):
    """Per row: GPU window scores within tolerance of the oracle; the indices bit-exact against the
    oracle top-k of the GPU's own scores; >= 99.9% overlap with the oracle's own top-k."""
    kdec = decode(wl.k)
    expect = np.full((len(rows), wl.topk), -1, np.int32)
    for r, t in enumerate(rows):
        lo, hi = window(wl, int(t))
        g = gpu_rows[r].astype(np.float64)
        if hi > lo:
            o = ref.row(r)
            assert not np.any(np.isnan(g)), f"row {t}: NaN in window"
            b = tolerance_row(wl, int(t), lo, hi, kdec=kdec)
            assert np.all(np.abs(g - o) <= b), f"row {t}: score outside tolerance"
            sel = O.topk_dense(gpu_rows[r][None, :].astype(np.float32), np.array([0], np.int32),
                               np.array([hi - lo], np.int32), wl.topk)[0]
            expect[r] = np.where(sel >= 0, sel + lo, -1)
    assert np.array_equal(idx_rows, expect)
    ov = overlap(idx_rows, O.topk(ref, wl.topk))
    assert ov >= 0.999, ov
