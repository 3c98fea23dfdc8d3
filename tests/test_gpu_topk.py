"""dsa_topk against the oracle top-k on the same fp32 logits (bit-exact indices)."""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def run_topk(dsa, logits, ks, ke, k):
    import torch

    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    idx = dsa.topk(lg, torch.from_numpy(ks).cuda(), torch.from_numpy(ke).cuda(), k)
    assert dsa.get_device_error() == 0
    return idx.cpu().numpy()


def windows(rng, T, N):
    ks = rng.integers(-5, N, T).astype(np.int32)
    ke = (ks + rng.integers(-3, N + 5, T)).astype(np.int32)
    ks[0], ke[0] = 0, N  # full row
    ks[1], ke[1] = 5, 5  # empty
    ks[2], ke[2] = -10, 3  # starts before 0
    ks[3], ke[3] = N - 2, N + 100  # ends past N
    return ks, ke


@pytest.mark.parametrize("k", [1, 7, 64, 500, 2048])
def test_random_rows(dsa, k):
    rng = np.random.default_rng(k)
    T, N = 41, 3001
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ks, ke = windows(rng, T, N)
    got = run_topk(dsa, logits, ks, ke, k)
    assert np.array_equal(got, O.topk_dense(logits, ks, ke, k))


@pytest.mark.parametrize("T", [1500, 2000])
def test_more_rows_than_resident_ctas(dsa, T):
    """More rows than the streaming kernel's resident CTAs (six per SM), so every CTA walks
    several rows and the last round is partial (1500 and 2000 rows over 912 CTAs).  Causal-like
    windows (growing with the row) plus random ones, every row against the oracle."""
    rng = np.random.default_rng(T)
    N, k = 3000, 512
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ks, ke = windows(rng, T, N)
    grow = np.arange(T) % 3 == 0
    ks[grow] = 0
    ke[grow] = (np.arange(T)[grow] * N // T + 1).astype(np.int32)
    got = run_topk(dsa, logits, ks, ke, k)
    assert np.array_equal(got, O.topk_dense(logits, ks, ke, k))


def test_ties_and_signed_zeros(dsa):
    rng = np.random.default_rng(1)
    T, N = 23, 1500
    levels = np.array([-1.0, -0.0, 0.0, 1.0, 2.5], dtype=np.float32)
    logits = levels[rng.integers(0, len(levels), (T, N))]
    ks, ke = windows(rng, T, N)
    for k in (1, 100, 333, 1000):
        assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


@pytest.mark.parametrize("spread,levels", [(2.0 ** -6, 0), (2.0 ** -10, 0), (2.0 ** -16, 0), (2.0 ** -10, 40)])
def test_close_scores_refine_threshold_bin(dsa, spread, levels):
    """Scores packed into a narrow band share their top 16 (or 24) key bits, so the threshold bin
    of the two-digit select holds far more keys than can be ranked directly: the select refines it
    digit by digit; with only `levels` distinct values near the threshold it ends in exact ties."""
    rng = np.random.default_rng(int(1 / spread) + levels)
    T, N = 19, 6000
    if levels:
        logits = (1.0 + spread * rng.integers(0, levels, (T, N)) / levels).astype(np.float32)
    else:
        logits = (1.0 + spread * rng.random((T, N))).astype(np.float32)
    ks, ke = windows(rng, T, N)
    for k in (7, 500, 2048):
        assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


def test_every_window_alignment_and_short_windows(dsa):
    """Windows starting at every offset modulo 4 keys, of every length from 1 to 40, with k below
    and above the length: the staged copy of a row covers its 16-byte aligned interior and the
    keys before and after it are read separately."""
    rng = np.random.default_rng(5)
    N = 1000
    starts, lens = np.meshgrid(np.arange(8), np.arange(1, 41))
    ks = (starts.ravel() * 37 + 3 * lens.ravel()).astype(np.int32)
    ke = (ks + lens.ravel()).astype(np.int32)
    T = len(ks)
    logits = rng.standard_normal((T, N)).astype(np.float32)
    for k in (1, 3, 17):
        assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


def test_logits_not_16_byte_aligned(dsa):
    """A logits pointer that is only 4-byte aligned takes the path without bulk copies."""
    import torch

    rng = np.random.default_rng(6)
    T, N, k = 9, 3000, 100
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ks, ke = windows(rng, T, N)
    flat = torch.from_numpy(np.concatenate([[0.0], logits.ravel()]).astype(np.float32)).cuda()
    lg = flat[1:].view(T, N)  # 4 bytes past a 16-byte boundary
    assert lg.data_ptr() % 16 == 4
    idx = dsa.topk(lg, torch.from_numpy(ks).cuda(), torch.from_numpy(ke).cuda(), k)
    assert dsa.get_device_error() == 0
    assert np.array_equal(idx.cpu().numpy(), O.topk_dense(logits, ks, ke, k))


def test_all_equal_rows(dsa):
    T, N = 4, 5000
    logits = np.full((T, N), 0.25, dtype=np.float32)
    ks = np.array([0, 10, 100, 4000], np.int32)
    ke = np.array([N, 4000, 4999, N], np.int32)
    for k in (1, 999, 2048):
        assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


def test_out_of_window_values_are_never_read(dsa):
    """NaN outside every window must not change the result (the kernel reads windows only)."""
    rng = np.random.default_rng(2)
    T, N = 16, 2000
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ks, ke = windows(rng, T, N)
    poisoned = logits.copy()
    for t in range(T):
        lo, hi = max(0, min(ks[t], N)), max(0, min(ke[t], N))
        poisoned[t, :lo] = np.nan
        poisoned[t, max(lo, hi):] = np.nan
    assert np.array_equal(run_topk(dsa, poisoned, ks, ke, 300), O.topk_dense(logits, ks, ke, 300))


def test_window_sizes_around_k(dsa):
    N, k = 4096, 512
    sizes = [0, 1, k - 1, k, k + 1, 2 * k, N]
    T = len(sizes)
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ks = np.zeros(T, np.int32)
    ke = np.array(sizes, np.int32)
    assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


def test_rows_longer_than_the_shared_memory_cache(dsa):
    """70000-key rows exceed the key cache: those rows take the re-read path."""
    rng = np.random.default_rng(4)
    T, N = 3, 70000
    logits = (rng.standard_normal((T, N)) * 3).astype(np.float32)
    logits[1, ::7] = 1.5  # many ties
    ks = np.array([0, 100, 0], np.int32)
    ke = np.array([N, N, 60000], np.int32)
    assert np.array_equal(run_topk(dsa, logits, ks, ke, 2048), O.topk_dense(logits, ks, ke, 2048))


def test_extreme_magnitudes(dsa):
    T, N = 2, 3000
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((T, N)) * 1e30).astype(np.float32)
    logits[0, :100] = -3.0e38
    logits[1, 50:60] = np.float32(1e-40)  # subnormals
    logits[1, 60:70] = -np.float32(1e-40)
    ks = np.zeros(T, np.int32)
    ke = np.full(T, N, np.int32)
    assert np.array_equal(run_topk(dsa, logits, ks, ke, 1500), O.topk_dense(logits, ks, ke, 1500))


@pytest.mark.parametrize("k", [1, 3])
def test_tiny_windows_every_offset(dsa, k):
    """Windows of k+1 .. k+13 keys starting at every offset within a 4-key vector: the staged
    row's partial vectors at both ends (one vector holding the whole window, two partial ones,
    partial + whole + partial) are converted one key at a time, the whole ones without tests."""
    rng = np.random.default_rng(11 + k)
    N = 96
    starts, lens = np.meshgrid(np.arange(40, 48), np.arange(k + 1, k + 14))
    ks = starts.ravel().astype(np.int32)
    ke = (ks + lens.ravel()).astype(np.int32)
    T = len(ks)
    logits = rng.standard_normal((T, N)).astype(np.float32)
    logits[::3, 40:60] = 0.5  # ties inside the window, broken by the lower index
    assert np.array_equal(run_topk(dsa, logits, ks, ke, k), O.topk_dense(logits, ks, ke, k))


def test_refinement_sweep_ragged_ends(dsa):
    """Keys packed into one top-digit bin (the refinement sweep runs) over windows whose start
    and end fall at every offset within a 4-key vector."""
    rng = np.random.default_rng(12)
    N = 2000
    ks = np.repeat(np.arange(100, 104), 4).astype(np.int32)
    ke = (np.arange(1700, 1716) % 4 + 1700 + 4 * np.arange(16)).astype(np.int32)
    T = len(ks)
    logits = (1.0 + 2.0 ** -12 * rng.random((T, N))).astype(np.float32)
    assert np.array_equal(run_topk(dsa, logits, ks, ke, 700), O.topk_dense(logits, ks, ke, 700))
