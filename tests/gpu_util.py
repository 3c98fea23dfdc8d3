"""Helpers shared by the GPU parity tests: device copies, the score tolerance, comparisons.

The tolerance is the fp32 accumulation bound, in score units,
    B(t, j) = 1e-4 * |k_scale[j]| * sum_h |w[t, h]| * sum_d |q[t, h, d] k[j, d]| + 1e-6,
computed here in float64 from decoded inputs (torch's float8_e4m3fn decoder, independent of the
oracle and of the library).
"""
from __future__ import annotations

import numpy as np

import oracle as O


_E4M3 = None


def decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of e4m3 codes, by a 256-entry table taken from torch's float8_e4m3fn decoder."""
    global _E4M3
    if _E4M3 is None:
        import torch

        _E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
            torch.float64).numpy()
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


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


def tolerance_rows(wl, rows, kabs=None) -> np.ndarray:
    """B(t, j) for the listed rows and every key, float64 [R, N].

    sum_h |w[t,h]| sum_d |q[t,h,d]| |k[j,d]| = sum_d |k[j,d]| v[t,d] with v[t,d] = sum_h |w[t,h]| |q[t,h,d]|
    (all terms non-negative), so the bound of a whole slab of rows is one matrix product."""
    rows = np.asarray(rows, dtype=np.int64)
    kabs = np.abs(decode(wl.k)) if kabs is None else kabs
    v = np.einsum("rh,rhd->rd", np.abs(wl.w[rows].astype(np.float64)), np.abs(decode(wl.q[rows])))
    return 1e-4 * np.abs(wl.k_scale.astype(np.float64))[None, :] * (v @ kabs.T) + 1e-6


def check_scores(wl, logits_rows: np.ndarray, rows, ref: O.RowScores, exact=False, slab=512):
    """Every in-window GPU score of the listed rows within tolerance of the oracle (or equal).

    logits_rows[r] is the GPU logits row of token rows[r].  Checked a slab of rows at a time
    (dense [slab, N] arrays), so all rows of an 8192-token problem take seconds.  Returns the worst
    error / bound.
    """
    rows = np.asarray(rows, dtype=np.int64)
    worst = 0.0
    kabs = np.abs(decode(wl.k))
    cols = np.arange(wl.N, dtype=np.int64)[None, :]
    for s0 in range(0, len(rows), slab):
        rs = rows[s0:s0 + slab]
        lo = ref.lo[s0:s0 + slab].astype(np.int64)
        n = ref.length[s0:s0 + slab].astype(np.int64)
        mask = (cols >= lo[:, None]) & (cols < (lo + n)[:, None])
        g = np.asarray(logits_rows[s0:s0 + slab], dtype=np.float64)
        o = np.zeros_like(g)
        for r in range(len(rs)):
            if n[r] > 0:
                o[r, lo[r]:lo[r] + n[r]] = ref.row(s0 + r)
        nan = np.isnan(g) & mask
        if nan.any():
            r, j = np.argwhere(nan)[0]
            raise AssertionError(f"row {rs[r]}: NaN in window at key {j}")
        if exact:
            bad = mask & (g != o)
            if bad.any():
                r, j = np.argwhere(bad)[0]
                raise AssertionError(f"row {rs[r]}: {int(bad[r].sum())} inexact, first key {j}: {g[r, j]} vs {o[r, j]}")
        else:
            b = tolerance_rows(wl, rs, kabs=kabs)
            ratio = np.where(mask, np.abs(g - o) / b, 0.0)
            m = float(ratio.max()) if ratio.size else 0.0
            if not m <= 1.0:
                r, j = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
                raise AssertionError(f"row {rs[r]} key {j}: |{g[r, j]} - {o[r, j]}| > {b[r, j]}")
            worst = max(worst, m)
    return worst


def overlap(idx_a: np.ndarray, idx_b: np.ndarray) -> float:
    """sum_rows |A & B| / sum_rows |B| over valid (non -1) entries (set semantics per row)."""
    a = np.asarray(idx_a, dtype=np.int64)
    b = np.asarray(idx_b, dtype=np.int64)
    assert a.shape[0] == b.shape[0]
    R = a.shape[0]
    span = int(max(a.max(initial=-1), b.max(initial=-1))) + 1
    if span == 0:
        return 1.0
    inter = total = 0
    slab = max(1, (64 << 20) // span)  # rows per slab of [slab, span] presence maps
    for r0 in range(0, R, slab):
        sa, sb = a[r0:r0 + slab], b[r0:r0 + slab]
        ma = np.zeros((sa.shape[0], span), dtype=bool)
        mb = np.zeros((sb.shape[0], span), dtype=bool)
        ra, ca = np.nonzero(sa >= 0)
        rb, cb = np.nonzero(sb >= 0)
        ma[ra, sa[ra, ca]] = True
        mb[rb, sb[rb, cb]] = True
        inter += int(np.count_nonzero(ma & mb))
        total += int(np.count_nonzero(mb))
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
