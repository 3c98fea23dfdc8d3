"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes an oracle library handle (the real one, or a copy with a planted
mistake) and raises ``AssertionError`` when the oracle disagrees with what the pages and the
mathematics fix:

* the e4m3 format definition (spot values) and an independent decoder (torch's
  ``float8_e4m3fn``);
* a hand-computed worked example (``golden/worked_example.json``);
* brute force over all key subsets for the top-k rule;
* the special case that reduces to a library matrix product (numpy);
* exact rational arithmetic on integer-valued inputs;
* invariants: relu sign, key permutation, power-of-two scaling, window restriction, -1
  padding of short windows;
* the key quantiser: round trip of every code, torch's float8_e4m3fn rounding, exact midpoints
  (ties to even) and saturation, and per-row properties (the largest magnitude lands on 448,
  the e4m3 error bound, zero rows, power-of-two and sign invariance);
* sparse attention: the plain mean of the listed rows (q = 0), scipy's softmax over the listed
  keys with the sink as an extra zero-valued logit, one listed key (logistic of s - sink), logits
  far past exp's range, and the multiset nature of the index list.
"""
from __future__ import annotations

import itertools
import json
import os
from fractions import Fraction

import numpy as np

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _decode_torch(codes: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _full_windows(T, N):
    return np.zeros(T, np.int32), np.full(T, N, np.int32)


# ----------------------------------------------------------------------------- e4m3


def pin_e4m3_spot(lib):
    """Values fixed by the E4M3FN definition: bias 7, 3 mantissa bits, max 448, no inf."""
    t = O.e4m3_table(lib)
    expect = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0xB8: -1.0, 0xC8: -4.0, 0x7E: 448.0, 0xFE: -448.0,
              0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x00: 0.0, 0x3C: 1.5, 0x77: 240.0}
    for c, v in expect.items():
        assert t[c] == v, (hex(c), t[c], v)
    assert np.signbit(t[0x80]) and t[0x80] == 0.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[0x00:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must increase"
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])


def pin_e4m3_torch(lib):
    """All 256 codes against torch's independent float8_e4m3fn decoder."""
    t = O.e4m3_table(lib)
    ref = _decode_torch(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.array_equal(t[~nan], ref[~nan])
    assert np.array_equal(np.signbit(t[~nan]), np.signbit(ref[~nan]))


# ----------------------------------------------------------------------------- worked example


def _worked():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        return json.load(f)


def _worked_inputs(g, pad_h=None, pad_d=None):
    q = np.array(g["q_codes"], np.uint8)
    w = np.array(g["w"], np.float32)
    k = np.array(g["k_codes"], np.uint8)
    kscale = np.array(g["k_scale"], np.float32)
    if pad_d:
        q = np.concatenate([q, np.zeros(q.shape[:2] + (pad_d - q.shape[2],), np.uint8)], axis=2)
        k = np.concatenate([k, np.zeros((k.shape[0], pad_d - k.shape[1]), np.uint8)], axis=1)
    if pad_h:
        T, H, D = q.shape
        q = np.concatenate([q, np.full((T, pad_h - H, D), 0x38, np.uint8)], axis=1)  # nonzero q rows ...
        w = np.concatenate([w, np.zeros((T, pad_h - H), np.float32)], axis=1)  # ... with zero weight
    ks = np.array([g["token0"]["ks"], g["token1"]["ks"]], np.int32)
    ke = np.array([g["token0"]["ke"], g["token1"]["ke"]], np.int32)
    return q, w, k, kscale, ks, ke


def _check_worked(lib, q, w, k, kscale, ks, ke, g):
    sc = O.index_score(q, w, k, kscale, ks, ke, lib=lib, nthreads=1)
    assert np.array_equal(sc.row(0), np.array(g["scores"])), sc.row(0)
    assert list(sc.row(1)) == g["scores"][1:3], sc.row(1)
    for tok, r in (("token0", 0), ("token1", 1)):
        for kk, expect in g[tok]["topk"].items():
            kk = int(kk)
            sub = O.RowScores(rows=sc.rows[r:r + 1], lo=sc.lo[r:r + 1], length=sc.length[r:r + 1],
                              offsets=np.zeros(1, np.int64), flat=sc.row(r).copy())
            got = O.topk(sub, kk, lib=lib, nthreads=1)[0].tolist()
            assert got == expect, (tok, kk, got, expect)


def pin_worked_example(lib):
    g = _worked()
    codes = g["e4m3_codes"]
    tab = O.e4m3_table(lib)
    for v, c in codes.items():
        assert tab[c] == float(v)
    _check_worked(lib, *_worked_inputs(g), g)


def pin_worked_example_padded(lib):
    """Zero-padding D and adding zero-weight heads leaves every score and selection unchanged."""
    g = _worked()
    _check_worked(lib, *_worked_inputs(g, pad_h=4, pad_d=64), g)


# ----------------------------------------------------------------------------- top-k rule


def _brute_topk(vals, lo, hi, k):
    """Unique S, |S| = min(k, n), such that each member beats each non-member under
    (larger score, then lower index); returned ascending and -1 padded."""
    keys = list(range(lo, hi))
    m = min(k, len(keys))
    found = []
    for S in itertools.combinations(keys, m):
        Sset = set(S)
        ok = all((vals[s] > vals[o]) or (vals[s] == vals[o] and s < o)
                 for s in S for o in keys if o not in Sset)
        if ok:
            found.append(sorted(S))
    assert len(found) == 1, found
    return found[0] + [-1] * (k - m)


def pin_topk_bruteforce(lib):
    rng = np.random.default_rng(7)
    levels = np.array([-1.0, -0.0, 0.0, 0.5, 1.0, 2.0, -3.5])
    for trial in range(60):
        N = int(rng.integers(1, 9))
        vals = levels[rng.integers(0, len(levels), N)] if trial % 2 == 0 else rng.standard_normal(N)
        lo = int(rng.integers(0, N))
        hi = int(rng.integers(lo, N + 1))
        for k in range(1, N + 3):
            expect = _brute_topk(vals, lo, hi, k)
            got = O.topk_dense(vals[None, :], np.array([lo]), np.array([hi]), k, lib=lib, nthreads=1)[0]
            assert got.tolist() == expect, (vals, lo, hi, k, got, expect)
            got32 = O.topk_dense(vals[None, :].astype(np.float32), np.array([lo]), np.array([hi]), k, lib=lib,
                                 nthreads=1)[0]
            assert got32.tolist() == expect


# ----------------------------------------------------------------------------- closed forms


def pin_closed_form_matmul(lib):
    """H = 1, w = 1, k_scale = 1, q, k >= 0: relu is inactive and score = K @ q (numpy)."""
    T, N, D = 3, 50, 32
    q_codes = W.encode_e4m3(np.abs(W.normal(11, 1, T * D)) * 3).reshape(T, 1, D)
    k_codes = W.encode_e4m3(np.abs(W.normal(11, 2, N * D)) * 3).reshape(N, D)
    ks, ke = _full_windows(T, N)
    sc = O.index_score(q_codes, np.ones((T, 1), np.float32), k_codes, np.ones(N, np.float32), ks, ke, lib=lib,
                       nthreads=1)
    ref = _decode_torch(k_codes) @ _decode_torch(q_codes[:, 0, :]).T  # [N, T]
    for t in range(T):
        np.testing.assert_allclose(sc.row(t), ref[:, t], rtol=1e-13, atol=0)
    # and with signs: H = 1, w = 1 -> relu(K @ q) * k_scale
    q2 = W.encode_e4m3(W.normal(12, 1, T * D)).reshape(T, 1, D)
    kscale = (np.arange(N) % 5 + 1).astype(np.float32) * 0.25
    sc2 = O.index_score(q2, np.ones((T, 1), np.float32), k_codes, kscale, ks, ke, lib=lib, nthreads=1)
    ref2 = np.maximum(_decode_torch(k_codes) @ _decode_torch(q2[:, 0, :]).T, 0.0) * kscale[:, None]
    for t in range(T):
        np.testing.assert_allclose(sc2.row(t), ref2[:, t], rtol=1e-13, atol=1e-300)


def pin_integer_exact(lib):
    """Integer q, k in [-4, 4], w in {+-0.5, +-1, +-2}, k_scale in {0.5, 1, 2}: every quantity is
    an exact binary fraction, so the double result equals exact rational arithmetic."""
    T, N, H, D = 6, 40, 3, 8
    ks = np.array([0, 3, 10, -3, 39, 5], np.int32)
    ke = np.array([40, 17, 10, 1, 40, 60], np.int32)  # empty window, negative start, end past N
    wl = W.make_integer("int", T, N, H, D, 5, 21, ks, ke)
    qi = _decode_torch(wl.q).astype(np.int64)
    ki = _decode_torch(wl.k).astype(np.int64)
    assert np.array_equal(qi, _decode_torch(wl.q)) and np.abs(qi).max() <= 4
    sc = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, ks, ke, lib=lib, nthreads=1)
    for t in range(T):
        lo, hi = max(0, min(int(ks[t]), N)), max(0, min(int(ke[t]), N))
        assert int(sc.lo[t]) == lo and int(sc.length[t]) == max(0, hi - lo)
        got = sc.row(t)
        for j in range(lo, hi):
            acc = Fraction(0)
            for h in range(H):
                dot = int(np.dot(qi[t, h], ki[j]))
                acc += Fraction(max(dot, 0)) * Fraction(float(wl.w[t, h]))
            exact = acc * Fraction(float(wl.k_scale[j]))
            assert Fraction(float(got[j - lo])) == exact, (t, j, got[j - lo], exact)


# ----------------------------------------------------------------------------- invariants


def _small_normal(seed=5, T=5, N=64, H=4, D=16):
    ks, ke = _full_windows(T, N)
    return W.make_normal("pin", T, N, H, D, 8, seed, ks, ke)


def pin_relu_sign(lib):
    """w >= 0 gives scores >= 0 and w <= 0 gives scores <= 0, although many dots are negative."""
    wl = _small_normal()
    for sign in (1.0, -1.0):
        w = (np.abs(wl.w) * sign).astype(np.float32)
        sc = O.index_score(wl.q, w, wl.k, wl.k_scale, wl.ks, wl.ke, lib=lib, nthreads=1)
        assert np.all(sc.flat * sign >= 0.0), sign
        assert np.count_nonzero(sc.flat) > len(sc.flat) // 2  # not trivially zero


def pin_permutation(lib):
    """Permuting the keys permutes the scores.  The multiset of selected scores never changes,
    and the selected key set maps back to the same keys whenever the k-th and (k+1)-th largest
    scores differ (otherwise the tie rule picks by position, which the permutation moves)."""
    wl = _small_normal(seed=6)
    perm = np.random.default_rng(3).permutation(wl.N)
    base = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, lib=lib, nthreads=1)
    per = O.index_score(wl.q, wl.w, wl.k[perm], wl.k_scale[perm], wl.ks, wl.ke, lib=lib, nthreads=1)
    for t in range(wl.T):
        assert np.array_equal(per.row(t), base.row(t)[perm])
    checked_sets = 0
    for kk in (1, 7, 30, wl.N):
        a = O.topk(base, kk, lib=lib, nthreads=1)
        b = O.topk(per, kk, lib=lib, nthreads=1)
        for t in range(wl.T):
            ra, rb = base.row(t), per.row(t)
            sa = [x for x in a[t].tolist() if x >= 0]
            sb = [x for x in b[t].tolist() if x >= 0]
            assert sorted(ra[sa].tolist()) == sorted(rb[sb].tolist())
            desc = np.sort(ra)[::-1]
            if kk >= wl.N or desc[kk - 1] != desc[kk]:
                assert sorted(sa) == sorted(int(perm[x]) for x in sb)
                checked_sets += 1
    assert checked_sets >= 10


def pin_pow2_scaling(lib):
    """Scaling w or k_scale by a power of two scales every score exactly; selection unchanged."""
    wl = _small_normal(seed=8)
    base = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, lib=lib, nthreads=1)
    s1 = O.index_score(wl.q, (wl.w * 4).astype(np.float32), wl.k, wl.k_scale, wl.ks, wl.ke, lib=lib, nthreads=1)
    s2 = O.index_score(wl.q, wl.w, wl.k, (wl.k_scale * 0.125).astype(np.float32), wl.ks, wl.ke, lib=lib,
                       nthreads=1)
    assert np.array_equal(s1.flat, base.flat * 4)
    assert np.array_equal(s2.flat, base.flat * 0.125)
    for s in (s1, s2):
        assert np.array_equal(O.topk(s, 9, lib=lib), O.topk(base, 9, lib=lib))


def pin_window_restriction(lib):
    """A sub-window changes no score; its top-k is the full-row top-k rule applied to the sub-window."""
    wl = _small_normal(seed=9)
    full = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, lib=lib, nthreads=1)
    ks2 = np.array([3, 0, 20, 63, 10], np.int32)
    ke2 = np.array([40, 64, 21, 64, 10], np.int32)
    sub = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, ks2, ke2, lib=lib, nthreads=1)
    dense = full.dense(wl.N)
    for t in range(wl.T):
        assert np.array_equal(sub.row(t), dense[t, ks2[t]:ke2[t]])
    for kk in (1, 5, 17):
        assert np.array_equal(O.topk(sub, kk, lib=lib), O.topk_dense(dense, ks2, ke2, kk, lib=lib))


def pin_short_window_padding(lib):
    """A window shorter than k returns every key of the window in ascending order, then -1."""
    wl = _small_normal(seed=10)
    ks2 = np.array([0, 5, 30, -5, 70], np.int32)
    ke2 = np.array([3, 6, 30, 2, 80], np.int32)  # 3 keys, 1 key, empty, negative start, past N
    sc = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, ks2, ke2, lib=lib, nthreads=1)
    idx = O.topk(sc, 8, lib=lib)
    assert idx[0].tolist() == [0, 1, 2] + [-1] * 5
    assert idx[1].tolist() == [5] + [-1] * 7
    assert idx[3].tolist() == [0, 1] + [-1] * 6
    for r in (2, 4):
        assert idx[r].tolist() == [-1] * 8


# ----------------------------------------------------------------------------- key quantiser


def pin_e4m3_encode_roundtrip(lib):
    """Every finite code's value encodes back to that code (the nearest value is itself)."""
    t = O.e4m3_table(lib)
    codes = np.arange(256, dtype=np.uint8)
    fin = ~np.isnan(t)
    assert np.array_equal(O.e4m3_encode(t[fin].astype(np.float32), lib=lib), codes[fin])


def pin_e4m3_encode_torch(lib):
    """Against torch's independent float32 -> float8_e4m3fn rounding (round to nearest even), on
    magnitudes up to 448."""
    import torch

    rng = np.random.default_rng(17)
    y = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)]).astype(np.float32)
    y = y[np.abs(y) <= 448.0]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(y, lib=lib)
    assert np.array_equal(got, ref), int(np.sum(got != ref))


def pin_e4m3_ties_and_saturation(lib):
    """Midpoints between neighbouring values go to the even code; the float just above or below a
    midpoint goes to the nearer value; magnitudes beyond 448 saturate; the sign is kept."""
    t = O.e4m3_table(lib)
    pos = t[0x00:0x7F]
    for c in range(0, 0x7E):
        mid = (pos[c] + pos[c + 1]) / 2
        assert np.float32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        ys = np.array([mid, np.nextafter(np.float32(mid), np.float32(0)), np.nextafter(np.float32(mid), np.float32(1e9)),
                       -mid], np.float32)
        got = O.e4m3_encode(ys, lib=lib)
        assert got.tolist() == [even, c, c + 1, 0x80 | even], (c, got)
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, -500.0, -1e30], np.float32)
    assert O.e4m3_encode(big, lib=lib).tolist() == [0x7E] * 5 + [0xFE, 0xFE]
    assert O.e4m3_encode(np.array([0.0, -0.0, 1e-30, -1e-30], np.float32), lib=lib).tolist() == [0, 0x80, 0, 0x80]


def _bf16_rows(rng, N, D, scales):
    x = (rng.standard_normal((N, D)) * scales[:, None]).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation to bf16 (any bf16 value will do)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def pin_quantize_rows(lib):
    """Per row: the largest magnitude encodes to +-448; every value is reproduced within half an
    e4m3 step (relative 2^-4 in the normal range, 2^-10 s below it); zero rows give scale 0 and
    code 0."""
    rng = np.random.default_rng(23)
    N, D = 300, 64
    bits, vals = _bf16_rows(rng, N, D, 10.0 ** rng.uniform(-6, 6, N))
    bits[7] = 0
    bits[8] = 0x8000  # -0.0
    vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scale = O.quantize_rows(bits, lib=lib)
    t = O.e4m3_table(lib)
    for r in range(N):
        m = np.max(np.abs(vals[r]))
        if m == 0:
            assert scale[r] == 0 and np.all(codes[r] == 0), r
            continue
        s = float(scale[r])
        assert abs(s - m / 448) <= 1e-6 * m / 448, r
        top = int(np.argmax(np.abs(vals[r])))
        assert codes[r, top] == (0xFE if vals[r, top] < 0 else 0x7E), r
        deq = t[codes[r]] * s
        err = np.abs(deq - vals[r])
        bound = np.maximum(np.abs(vals[r]) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6)
        assert np.all(err <= bound), (r, float(np.max(err / bound)))


def pin_quantize_invariants(lib):
    """Scaling a row by a power of two scales its scale alike and keeps its codes; negating it
    flips every code's sign bit (except for zeros, whose code keeps the input's sign)."""
    rng = np.random.default_rng(29)
    bits, vals = _bf16_rows(rng, 64, 128, 10.0 ** rng.uniform(-3, 3, 64))
    codes, scale = O.quantize_rows(bits, lib=lib)
    for p in (-5, 3):
        b2 = ((vals * np.float32(2.0 ** p)).view(np.uint32) >> 16).astype(np.uint16)
        c2, s2 = O.quantize_rows(b2, lib=lib)
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2, (scale * np.float32(2.0 ** p)).astype(np.float32))
    cn, sn = O.quantize_rows(bits ^ np.uint16(0x8000), lib=lib)
    assert np.array_equal(sn, scale)
    assert np.array_equal(cn, codes ^ np.uint8(0x80))


# ---------------------------------------------------------------------- sparse attention


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values that bf16 holds exactly (asserted)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, x), "value not exact in bf16"
    return bits


def _attn_case(seed, T=5, N=23, H=3, D=8, K=9, span=8):
    """bf16-exact q / kv (multiples of 1/8 in [-span, span]), index lists with -1 entries and
    repeated keys."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-8 * span, 8 * span + 1, (T, H, D)) / 8.0
    kv = rng.integers(-8 * span, 8 * span + 1, (N, D)) / 8.0
    idx = rng.integers(-1, N, (T, K)).astype(np.int32)
    idx[0, :3] = [4, 4, 9]  # a repeated key
    idx[1, :] = -1
    idx[1, 5] = 7  # one key
    idx[2, :] = -1  # none
    return q, kv, idx


def _attn_dense(q, kv, sink, idx, scale):
    """The definition through library routines: numpy matrix products and scipy's softmax over
    the listed keys, the sink as one extra logit whose value row is zero."""
    from scipy.special import softmax

    T, H, D = q.shape
    out = np.zeros((T, H, D))
    for t in range(T):
        lst = idx[t][idx[t] >= 0]
        if len(lst) == 0:
            continue
        v = kv[lst]
        s = scale * (q[t] @ v.T)  # [H, L]
        if sink is not None:
            s = np.concatenate([s, np.asarray(sink, np.float64)[:, None]], axis=1)
            v = np.concatenate([v, np.zeros((1, D))], axis=0)
        out[t] = softmax(s, axis=1) @ v
    return out


def pin_attn_mean(lib):
    """q = 0 and no sink: every listed key weighs the same, so the output is the plain mean of
    the listed kv rows (a repeated key counted each time); an empty list gives 0."""
    _, kv, idx = _attn_case(21)
    q = np.zeros((idx.shape[0], 3, kv.shape[1]))
    got = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), None, idx, 0.7, lib=lib)
    for t in range(idx.shape[0]):
        lst = idx[t][idx[t] >= 0]
        want = kv[lst].mean(axis=0) if len(lst) else np.zeros(kv.shape[1])
        assert np.allclose(got[t], want[None, :], rtol=1e-13, atol=1e-13), t


def pin_attn_softmax_library(lib):
    """Random bf16-exact inputs, with and without a sink: the oracle equals scipy's softmax
    weights applied to the listed rows (the sink as an extra logit with a zero value row)."""
    for seed, sink in ((22, None), (23, np.array([0.5, -2.0, 3.25], np.float32))):
        q, kv, idx = _attn_case(seed, span=2)
        scale = 1.0 / np.sqrt(q.shape[2])
        got = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, idx, scale, lib=lib)
        want = _attn_dense(q, kv, sink, idx, scale)
        assert np.allclose(got, want, rtol=1e-11, atol=1e-12)


def pin_attn_single_key(lib):
    """One listed key j: without a sink the output is kv[j] exactly; with a sink it is
    kv[j] * logistic(s_j - sink) (scipy's expit)."""
    from scipy.special import expit

    q, kv, _ = _attn_case(24)
    idx = np.full((q.shape[0], 4), -1, np.int32)
    idx[:, 2] = np.arange(q.shape[0]) * 3 % kv.shape[0]
    sink = np.array([1.0, -0.5, 0.0], np.float32)
    scale = 0.05
    got = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), None, idx, scale, lib=lib)
    assert np.array_equal(got, np.broadcast_to(kv[idx[:, 2]][:, None, :], got.shape))
    got = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, idx, scale, lib=lib)
    for t in range(q.shape[0]):
        j = idx[t, 2]
        s = scale * (q[t] @ kv[j])
        want = kv[j][None, :] * expit(s - sink.astype(np.float64))[:, None]
        assert np.allclose(got[t], want, rtol=1e-13, atol=1e-15)


def pin_attn_large_logits(lib):
    """Logits spread over ~10^4 (far past exp's double range): the result stays finite and
    equals the library softmax, which shifts by the row maximum."""
    q, kv, idx = _attn_case(25, D=16, span=30)
    sink = np.array([5.0, 4000.0, -3.0], np.float32)
    for sk in (None, sink):
        got = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sk, idx, 1.0, lib=lib)
        assert np.all(np.isfinite(got))
        assert np.allclose(got, _attn_dense(q, kv, sk, idx, 1.0), rtol=1e-9, atol=1e-9)


def pin_attn_list_order(lib):
    """The output depends on the index list as a multiset: permuting its entries (the -1 ones
    included) changes nothing; out-of-range indices are rejected."""
    q, kv, idx = _attn_case(26, span=2)
    sink = np.array([0.25, 0.0, -1.0], np.float32)
    a = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, idx, 0.3, lib=lib)
    rng = np.random.default_rng(7)
    perm = np.stack([rng.permutation(row) for row in idx])
    b = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, perm, 0.3, lib=lib)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)
    bad = idx.copy()
    bad[3, 0] = kv.shape[0]
    try:
        O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, bad, 0.3, lib=lib)
    except ValueError:
        pass
    else:
        raise AssertionError("an index past the last key was accepted")


def _bwd_case(seed, T=3, N=6, H=2, D=4, K=4):
    """Inputs whose entries are +-(1 + m/128), m in [1, 126]: exact in bf16, and a step of
    2^-7 either way stays exact (the finite differences below move one entry by that step)."""
    rng = np.random.default_rng(seed)

    def vals(shape):
        return rng.choice([-1.0, 1.0], shape) * (1.0 + rng.integers(1, 127, shape) / 128.0)

    q, kv, do = vals((T, H, D)), vals((N, D)), vals((T, H, D))
    idx = rng.integers(0, N, (T, K)).astype(np.int32)
    idx[0, :2] = [3, 3]  # a repeated key
    idx[1, 1] = -1
    return q, kv, do, idx


def _loss(q, kv, sink, idx, do, scale, lib):
    """sum(do * o) through the oracle's forward (the quantity the gradients are of)."""
    o = O.sparse_attn(_bf16_bits(q), _bf16_bits(kv), sink, idx, scale, lib=lib)
    return float(np.sum(do * o))


def pin_attn_bwd_finite_differences(lib):
    """Every entry of dq, dkv and dsink against a central difference of the forward oracle's
    loss sum(do * o) (q and kv moved by one bf16 step, 2^-7; the sink by 2^-10), with and
    without a sink, a repeated key and a -1 entry included."""
    q, kv, do, idx = _bwd_case(31)
    scale = 0.25
    for sink in (None, np.array([0.5, -0.75], np.float32)):
        dq, dkv, dsink = O.sparse_attn_bwd(_bf16_bits(q), _bf16_bits(kv), sink, idx, _bf16_bits(do), scale, lib=lib)
        e = 2.0 ** -7
        for arr, grad in ((q, dq), (kv, dkv)):
            for pos in np.ndindex(arr.shape):
                keep = arr[pos]
                arr[pos] = keep + e
                up = _loss(q, kv, sink, idx, do, scale, lib)
                arr[pos] = keep - e
                dn = _loss(q, kv, sink, idx, do, scale, lib)
                arr[pos] = keep
                fd = (up - dn) / (2 * e)
                assert abs(fd - grad[pos]) <= 1e-4 * (1.0 + abs(grad[pos])), (pos, fd, grad[pos])
        if sink is not None:
            for h in range(len(sink)):
                es = 2.0 ** -10
                s2 = sink.astype(np.float64).copy()
                s2[h] += es
                up = _loss(q, kv, s2.astype(np.float32), idx, do, scale, lib)
                s2[h] -= 2 * es
                dn = _loss(q, kv, s2.astype(np.float32), idx, do, scale, lib)
                fd = (up - dn) / (2 * es)
                assert abs(fd - dsink[h]) <= 1e-4 * (1.0 + abs(dsink[h])), (h, fd, dsink[h])
        else:
            assert dsink is None


def pin_attn_bwd_single_key(lib):
    """One listed key j per row: without a sink p = 1, so dq = 0 and dkv[j] is the sum of the
    rows' do; with a sink p = logistic(s_j - sink) (scipy's expit) and the gradients follow in
    closed form: dq = scale p (1 - p) dP kv_j, dkv_j += scale p (1 - p) dP q + p do,
    dsink = -p (1 - p) dP, with dP = do . kv_j."""
    from scipy.special import expit

    q, kv, do, _ = _bwd_case(32, T=4, N=5, H=2, D=4)
    idx = np.full((4, 3), -1, np.int32)
    idx[:, 1] = [2, 0, 2, 4]
    scale = 0.3
    dq, dkv, _ = O.sparse_attn_bwd(_bf16_bits(q), _bf16_bits(kv), None, idx, _bf16_bits(do), scale, lib=lib)
    assert np.array_equal(dq, np.zeros_like(dq))
    want = np.zeros_like(kv)
    for t in range(4):
        want[idx[t, 1]] += do[t].sum(axis=0)
    assert np.allclose(dkv, want, rtol=1e-13, atol=1e-13)
    sink = np.array([0.25, -1.5], np.float32)
    dq, dkv, dsink = O.sparse_attn_bwd(_bf16_bits(q), _bf16_bits(kv), sink, idx, _bf16_bits(do), scale, lib=lib)
    wq, wkv, ws = np.zeros_like(q), np.zeros_like(kv), np.zeros(2)
    for t in range(4):
        j = idx[t, 1]
        for h in range(2):
            p = expit(scale * (q[t, h] @ kv[j]) - float(sink[h]))
            dp = do[t, h] @ kv[j]
            g = p * (1 - p) * dp
            wq[t, h] = scale * g * kv[j]
            wkv[j] += scale * g * q[t, h] + p * do[t, h]
            ws[h] += -g
    assert np.allclose(dq, wq, rtol=1e-12, atol=1e-13)
    assert np.allclose(dkv, wkv, rtol=1e-12, atol=1e-13)
    assert np.allclose(dsink, ws, rtol=1e-12, atol=1e-13)


def pin_attn_bwd_sums(lib):
    """Without a sink the weights of a row sum to 1 and the ds_j to 0, so summed over all keys
    dkv equals the sum of do over the rows (and heads) that list any key; a row that lists one
    key several times has dq = 0.  Gradients are linear in do."""
    q, kv, do, idx = _bwd_case(33, T=5, N=9, H=3, D=8, K=6)
    idx[2, :] = 4  # one key, listed six times
    idx[3, :] = -1  # none
    scale = 0.2
    dq, dkv, _ = O.sparse_attn_bwd(_bf16_bits(q), _bf16_bits(kv), None, idx, _bf16_bits(do), scale, lib=lib)
    rows = [t for t in range(idx.shape[0]) if np.any(idx[t] >= 0)]
    assert np.allclose(dkv.sum(axis=0), do[rows].sum(axis=(0, 1)), rtol=1e-12, atol=1e-12)
    assert np.allclose(dq[2], 0.0, atol=1e-14) and np.array_equal(dq[3], np.zeros_like(dq[3]))
    dq2, dkv2, _ = O.sparse_attn_bwd(_bf16_bits(q), _bf16_bits(kv), None, idx, _bf16_bits(2 * do), scale, lib=lib)
    assert np.allclose(dq2, 2 * dq, rtol=1e-13, atol=1e-14) and np.allclose(dkv2, 2 * dkv, rtol=1e-13, atol=1e-14)


ALL_PINS = [
    pin_e4m3_spot,
    pin_e4m3_torch,
    pin_worked_example,
    pin_worked_example_padded,
    pin_topk_bruteforce,
    pin_closed_form_matmul,
    pin_integer_exact,
    pin_relu_sign,
    pin_permutation,
    pin_pow2_scaling,
    pin_window_restriction,
    pin_short_window_padding,
    pin_e4m3_encode_roundtrip,
    pin_e4m3_encode_torch,
    pin_e4m3_ties_and_saturation,
    pin_quantize_rows,
    pin_quantize_invariants,
    pin_attn_mean,
    pin_attn_softmax_library,
    pin_attn_single_key,
    pin_attn_large_logits,
    pin_attn_list_order,
    pin_attn_bwd_finite_differences,
    pin_attn_bwd_single_key,
    pin_attn_bwd_sums,
]
