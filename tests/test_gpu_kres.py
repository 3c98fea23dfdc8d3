"""dsa_index_score_kres (key tile resident, query blocks streamed) against the oracle and against
dsa_index_score (query block resident): the same scores bit for bit, only in-window entries
written, on integer inputs bit-exact against the oracle; workspace and alignment errors."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import check_scores, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def both(dsa, wl):
    import torch

    t = to_dev(wl)
    a = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    b = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    dsa.index_score(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=a)
    dsa.index_score_kres(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=b)
    assert dsa.get_device_error() == 0
    return a.cpu().numpy(), b.cpu().numpy()


def check(dsa, wl, exact=False):
    q_res, k_res = both(dsa, wl)
    # the same bits as the query-resident scorer, NaN fill kept in the same places
    assert np.array_equal(q_res.view(np.uint32), k_res.view(np.uint32))
    ref = O.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke)
    check_scores(wl, k_res, range(wl.T), ref, exact=exact)
    for t in range(wl.T):
        lo, n = int(ref.lo[t]), int(ref.length[t])
        assert np.all(np.isnan(k_res[t, :lo])) and np.all(np.isnan(k_res[t, lo + n:])), t


@pytest.mark.parametrize("H,D", [(4, 64), (64, 128), (32, 128), (8, 64), (16, 128), (64, 64), (4, 128)])
def test_integer_inputs_are_bit_exact(dsa, H, D):
    """Random (possibly empty, reversed or out-of-range) windows; several key tiles and token
    blocks with ragged tails."""
    T, N = 150, 333
    rng = np.random.default_rng(H * 1000 + D + 7)
    ks = rng.integers(-4, N, T).astype(np.int32)
    ke = (ks + rng.integers(-3, N, T)).astype(np.int32)
    wl = W.make_integer("int", T, N, H, D, 37, 7, ks, ke)
    check(dsa, wl, exact=True)


@pytest.mark.parametrize("H,D", [(4, 64), (32, 128), (64, 128), (16, 64)])
def test_normal_causal(dsa, H, D):
    T = 700  # more token blocks than one work item takes at these sizes
    ks, ke = W.causal_windows(T)
    wl = W.make_normal("causal", T, T, H, D, 64, 41 + H, ks, ke)
    check(dsa, wl)


def test_packed_documents(dsa):
    docs = (100, 700, 33, 1200)
    T = sum(docs)
    ks, ke = W.causal_windows(T, docs)
    wl = W.make_normal("docs", T, T, 64, 128, 128, 43, ks, ke, heavy_frac=0.01)
    check(dsa, wl)


def test_decode_like_windows(dsa):
    """One token per request over packed caches: each key tile meets one token's window."""
    wl = W.make_decode(seed=47, requests=24, lo=100, hi=3000, topk=64, H=16, D=128)
    check(dsa, wl)


def test_prefill_8192_tokens_equals_query_resident(dsa):
    """The 8192-token 64-head causal prefill at full size: bit-identical to dsa_index_score
    (which the configuration tests check against the oracle), and every 64th row against the
    oracle directly."""
    import torch

    wl = W.make_config("dsv32")
    t = to_dev(wl)
    a = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    b = torch.full((wl.T, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    dsa.index_score(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=a)
    dsa.index_score_kres(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], logits=b)
    assert dsa.get_device_error() == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    rows = np.arange(0, wl.T, 64)
    sub = W.Workload(**{**wl.__dict__, "T": len(rows), "q": wl.q[rows], "w": wl.w[rows], "ks": wl.ks[rows],
                        "ke": wl.ke[rows]})
    ref = O.index_score(sub.q, sub.w, sub.k, sub.k_scale, sub.ks, sub.ke)
    check_scores(sub, b[rows].cpu().numpy(), range(len(rows)), ref)


def test_workspace_and_alignment_errors(dsa):
    import torch

    wl = W.make_config("tiny")
    t = to_dev(wl)
    need = dsa.index_score_kres_workspace_size(wl.T, wl.N, wl.H, wl.D)
    assert need > 0
    short = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsa.DsaError, match="WORKSPACE"):
        dsa.index_score_kres(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], workspace=short)
    w_off = torch.empty(wl.T * wl.H + 1, dtype=torch.float32, device="cuda")[1:].view(wl.T, wl.H)
    w_off.copy_(t["w"])
    with pytest.raises(dsa.DsaError, match="INVALID_ARG"):
        dsa.index_score_kres(t["q"], w_off, t["k"], t["k_scale"], t["ks"], t["ke"])
    assert dsa.get_device_error() == 0
