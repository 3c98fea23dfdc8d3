"""dsa_index_score and dsa_index_topk against the oracle on small and ragged problems.

* scores: within B(t, j) of the oracle on every in-window pair, bit-exact on integer inputs;
* out-of-window logits are never written;
* fused top-k == dsa_topk(dsa_index_score(...)) bit for bit, and == the oracle top-k applied to
  the GPU's own scores; >= 99.9% overlap with the oracle's top-k of its own scores.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import check_scores, check_windowed, overlap, to_dev, windowed_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def gpu_all(dsa, wl, fill=np.nan):
    import torch

    t = to_dev(wl)
    logits = torch.full((wl.T, wl.N), fill, dtype=torch.float32, device="cuda")
    dsa.index_score(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=logits)
    idx_u = dsa.topk(logits, t["ks"], t["ke"], wl.topk)
    idx_f = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    return logits.cpu().numpy(), idx_u.cpu().numpy(), idx_f.cpu().numpy()


def full_check(dsa, wl, exact=False):
    logits, idx_u, idx_f = gpu_all(dsa, wl)
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke)
    check_scores(wl, logits, range(wl.T), ref, exact=exact)
    # out-of-window entries keep their NaN fill
    for t in range(wl.T):
        lo, n = int(ref.lo[t]), int(ref.length[t])
        assert np.all(np.isnan(logits[t, :lo])) and np.all(np.isnan(logits[t, lo + n:])), t
    expect = O.topk_dense(logits, wl.ks, wl.ke, wl.topk)
    assert np.array_equal(idx_u, expect)
    assert np.array_equal(idx_f, expect)
    ov = overlap(idx_f, O.topk(ref, wl.topk))
    if exact:
        assert ov == 1.0
    else:
        assert ov >= 0.999, ov
    return logits, idx_f


def windowed_check(dsa, wl):
    """full_check for problems whose [T, N] logits are too large to hold: every row's window is
    scored in slabs; fused indices against the oracle top-k of those GPU scores."""
    t = to_dev(wl)
    idx_f = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    rows = np.arange(wl.T)
    gpu_rows = windowed_scores(dsa, t, wl, rows)
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke)
    check_windowed(wl, rows, gpu_rows, ref, idx_f.cpu().numpy())


def causal(T, doc=None):
    return W.causal_windows(T, doc)


@pytest.mark.parametrize("H,D", [(4, 64), (64, 128), (32, 128), (8, 64), (16, 128), (64, 64), (4, 128)])
def test_integer_inputs_are_bit_exact(dsa, H, D):
    T, N = 150, 333
    rng = np.random.default_rng(H * 1000 + D)
    ks = rng.integers(-4, N, T).astype(np.int32)
    ke = (ks + rng.integers(0, N, T)).astype(np.int32)
    wl = W.make_integer("int", T, N, H, D, 37, 7, ks, ke)
    full_check(dsa, wl, exact=True)


@pytest.mark.parametrize("H,D,k", [(4, 64, 32), (32, 128, 64), (64, 128, 100), (16, 64, 16), (8, 128, 200)])
def test_normal_causal(dsa, H, D, k):
    T = 300
    ks, ke = causal(T)
    wl = W.make_normal("causal", T, T, H, D, k, 11 + H, ks, ke)
    full_check(dsa, wl)


def test_tiny_config(dsa):
    full_check(dsa, W.make_config("tiny"))


def test_glm_config(dsa):
    full_check(dsa, W.make_config("glm"))


def test_varlen_documents_small(dsa):
    docs = (100, 700, 33, 1200)
    T = sum(docs)
    ks, ke = causal(T, docs)
    wl = W.make_normal("docs", T, T, 64, 128, 128, 19, ks, ke, heavy_frac=0.01)
    full_check(dsa, wl)


def test_packed_decode_small(dsa):
    """Decode-like: 64 requests x 1 token, packed caches -> one token per unit, long rows split
    into chunks whose candidate lists are merged by the last chunk."""
    wl = W.make_decode(seed=31, requests=64, lo=500, hi=12000, topk=256)
    full_check(dsa, wl)


def test_decode_windows_not_aligned_to_tiles(dsa):
    lens = np.array([1, 127, 128, 129, 4095, 4097, 9000, 20000, 0, 3], np.int64)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    N = int(lens.sum())
    ks = starts.astype(np.int32)
    ke = (starts + lens).astype(np.int32)
    wl = W.make_normal("ragged", len(lens), N, 64, 128, 2048, 23, ks, ke)
    full_check(dsa, wl)


@pytest.mark.parametrize("lens,topk", [
    ((50000, 70000, 9000), 250),   # chunk lists merged in shared memory, topk not a multiple of 4
    ((30000, 20000, 12000, 5000), 2048),  # the same with 4-wide list loads
    ((300000,), 2048),             # more chunks than the staged merge takes: general list merge
    ((2_200_000,), 16),            # one very long row cut into about one chunk per SM
])
def test_split_rows_and_merges(dsa, lens, topk):
    """Rows longer than one item are cut into chunks whose candidate lists the last chunk merges;
    each merge path (staged in shared memory, scalar or 4-wide loads; general) against the oracle."""
    lens = np.asarray(lens, np.int64)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    N = int(lens.sum())
    ks = starts.astype(np.int32)
    ke = (starts + lens).astype(np.int32)
    wl = W.make_normal("split", len(lens), N, 4, 64, topk, 37 + len(lens), ks, ke)
    full_check(dsa, wl)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H", [4, 8, 16])
def test_long_causal_prefill_with_few_heads(dsa, H, D):
    """8192-token causal prefill with few heads: dsa_index_topk takes the scorer + selector route
    (faster than a fused unit of one or two tokens there).  Sampled rows against the oracle;
    the call's indices == dsa_topk(dsa_index_score()) on every row."""
    import torch

    T = N = 8192
    ks, ke = causal(T)
    wl = W.make_normal("fewheads", T, N, H, D, 2048, 53 + H + D, ks, ke)
    t = to_dev(wl)
    idx_f = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    logits = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    dsa.index_score(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=logits)
    idx_u = dsa.topk(logits, t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    idx_f = idx_f.cpu().numpy()
    assert np.array_equal(idx_u.cpu().numpy(), idx_f)
    rows = np.array(sorted(set(range(0, T, 251)) | {0, 1, 2047, 2048, 2049, T - 1}), np.int64)
    lg_rows = logits[torch.from_numpy(rows).cuda()].cpu().numpy()
    del logits
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows)
    check_scores(wl, lg_rows, rows, ref)
    assert np.array_equal(idx_f[rows], O.topk_dense(lg_rows, wl.ks[rows], wl.ke[rows], wl.topk))
    assert overlap(idx_f[rows], O.topk(ref, wl.topk)) >= 0.999


@pytest.mark.parametrize("H", [4, 16])
def test_few_heads_windows_longer_than_the_row_buffer(dsa, H):
    """Few heads with windows of 22-24K keys on a short query batch (the fused kernel, one token
    per unit): rows longer than the row buffer are cut into chunks and merged.  Every row against
    the oracle top-k of the GPU scores; fused == unfused."""
    import torch

    T, N = 256, 24576
    ks = np.zeros(T, np.int32)
    ke = (N - T + 1 + np.arange(T)).astype(np.int32)
    wl = W.make_normal("fewlong", T, N, H, 128, 2048, 71 + H, ks, ke)
    t = to_dev(wl)
    idx_f = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    logits = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
    dsa.index_score(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=logits)
    idx_u = dsa.topk(logits, t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    idx_f = idx_f.cpu().numpy()
    assert np.array_equal(idx_u.cpu().numpy(), idx_f)
    lg = logits.cpu().numpy()
    assert np.array_equal(idx_f, O.topk_dense(lg, wl.ks, wl.ke, wl.topk))
    rows = np.arange(0, T, 17, dtype=np.int64)
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows)
    check_scores(wl, lg[rows], rows, ref)
    assert overlap(idx_f[rows], O.topk(ref, wl.topk)) >= 0.999


def test_many_rows_longer_than_the_row_buffer(dsa):
    """More requests than SMs, each longer than a unit's shared-memory row buffer: units are cut
    into equal chunks under the capacity (not the few-long-rows split) and merged per row."""
    lens = np.full(160, 33_000, np.int64)
    lens[::7] = 70_001  # some rows need three chunks
    lens[5] = 0         # an empty request
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    N = int(lens.sum())
    wl = W.make_normal("long", len(lens), N, 4, 64, 512, 43, starts.astype(np.int32),
                       (starts + lens).astype(np.int32))
    windowed_check(dsa, wl)


def test_few_rows_split_exactly_and_short_rows(dsa):
    """Few rows: one row a whole number of split lengths long, one shorter than a split length,
    one shorter than k, and an empty one, together with long rows."""
    lens = np.array([4096 * 9, 4096 * 3, 3000, 100, 0, 250_000], np.int64)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    N = int(lens.sum())
    wl = W.make_normal("few", len(lens), N, 4, 64, 256, 47, starts.astype(np.int32),
                       (starts + lens).astype(np.int32))
    windowed_check(dsa, wl)


def test_empty_and_degenerate_windows(dsa):
    T, N = 70, 500
    ks = np.zeros(T, np.int32)
    ke = np.zeros(T, np.int32)
    ks[10:20], ke[10:20] = 5, 3  # ke < ks
    ks[20:30], ke[20:30] = 490, 900  # past N
    ks[30:40], ke[30:40] = -100, 7  # before 0
    ks[40:50], ke[40:50] = 0, N
    ks[50:], ke[50:] = 250, 251  # single key
    wl = W.make_normal("edge", T, N, 32, 128, 64, 29, ks, ke)
    full_check(dsa, wl)


def test_single_token_single_key(dsa):
    wl = W.make_normal("one", 1, 1, 4, 64, 1, 3, np.array([0], np.int32), np.array([1], np.int32))
    full_check(dsa, wl)


def test_no_keys(dsa):
    import torch

    T = 5
    wl = W.make_normal("nokeys", T, 0, 8, 64, 4, 3, np.zeros(T, np.int32), np.full(T, 3, np.int32))
    t = to_dev(wl)
    idx = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], 4)
    assert dsa.get_device_error() == 0
    assert np.array_equal(idx.cpu().numpy(), -np.ones((T, 4), np.int32))
    lg = torch.zeros((T, 0), dtype=torch.float32, device="cuda")
    idx2 = dsa.topk(lg, t["ks"], t["ke"], 4)
    assert np.array_equal(idx2.cpu().numpy(), -np.ones((T, 4), np.int32))


def test_repeated_calls_are_deterministic(dsa):
    wl = W.make_config("glm")
    _, a, b = gpu_all(dsa, wl)
    _, c, d = gpu_all(dsa, wl)
    assert np.array_equal(a, c) and np.array_equal(b, d)


def test_plan_reused_across_runs(dsa):
    """One plan, two runs with different q / w / k (as two layers sharing windows): each run
    equals a fresh dsa_index_topk, including rows merged from several chunks."""
    a = W.make_decode(seed=41, requests=64, lo=500, hi=12000, topk=256)
    b = W.make_decode(seed=41, requests=64, lo=500, hi=12000, topk=256)
    b2 = W.make_normal("layer2", a.T, a.N, a.H, a.D, a.topk, 99, a.ks, a.ke)
    ta, tb = to_dev(a), to_dev(b2)
    assert np.array_equal(a.ks, b.ks)
    ws = dsa.index_topk_plan(ta["ks"], ta["ke"], a.N, a.H, a.D, a.topk)
    r1 = dsa.index_topk_run(ta["q"], ta["w"], ta["k"], ta["k_scale"], ta["ks"], ta["ke"], a.topk, ws)
    r2 = dsa.index_topk_run(tb["q"], tb["w"], tb["k"], tb["k_scale"], tb["ks"], tb["ke"], a.topk, ws)
    r3 = dsa.index_topk_run(ta["q"], ta["w"], ta["k"], ta["k_scale"], ta["ks"], ta["ke"], a.topk, ws)
    f1 = dsa.index_topk(ta["q"], ta["w"], ta["k"], ta["k_scale"], ta["ks"], ta["ke"], a.topk)
    f2 = dsa.index_topk(tb["q"], tb["w"], tb["k"], tb["k_scale"], tb["ks"], tb["ke"], a.topk)
    assert dsa.get_device_error() == 0
    assert np.array_equal(r1.cpu().numpy(), f1.cpu().numpy())
    assert np.array_equal(r2.cpu().numpy(), f2.cpu().numpy())
    assert np.array_equal(r3.cpu().numpy(), f1.cpu().numpy())
    assert not np.array_equal(f1.cpu().numpy(), f2.cpu().numpy())


def test_workspace_too_small_is_rejected(dsa):
    import torch

    wl = W.make_config("tiny")
    t = to_dev(wl)
    need = dsa.index_topk_workspace_size(wl.T, wl.N, wl.H, wl.D, wl.topk)
    small = torch.empty(max(need - 256, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk, workspace=small)
    assert e.value.status == 3
