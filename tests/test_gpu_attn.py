"""dsa_sparse_attn against the oracle's sparse attention on the same seeded inputs.

The GPU computes in fp32 and rounds its output to bf16, so each (token, head) output vector is
checked against the oracle (double) within a bound derived from that arithmetic:
  * a score is a D-term fp32 dot product of exact products, times the scale: its error is at
    most E_s = D * 2^-24 * scale * sum_d |q[t,h,d]| * max|kv| (the running maximum carries the
    same bound);
  * each softmax weight then carries a relative error of at most 2 E_s + 8 * 2^-24 (expf and
    the subtraction), which moves the weighted mean of kv rows by at most twice that times
    max|kv|, and the fp32 accumulation over K listed rows adds K * 2^-24 * max|kv|;
  * the bf16 rounding of the output adds half an ulp, 2^-9 |o| (2^-8 |o| allowed);
  * the tensor-core kernel (D >= 128, H <= 64) rounds the softmax weights to bf16 before the
    weighted sum, as the DeepSeek V4.1 sparse_attn kernel casts them, while the denominator
    sums them in fp32: each weight's half-ulp, 2^-9 relative, moves the weighted mean by at most
    2^-9 max|kv| (2^-8 max|kv| allowed).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def _f(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gpu(dsa, q, kv, sink, idx, scale):
    import torch

    qt = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    kvt = torch.from_numpy(kv.view(np.int16)).cuda().view(torch.bfloat16)
    it = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    st = None if sink is None else torch.from_numpy(sink).cuda()
    out = dsa.sparse_attn(qt, kvt, it, attn_sink=st, scale=scale)
    assert dsa.get_device_error() == 0
    return _f(out.view(torch.int16).cpu().numpy().view(np.uint16))


def check(got, want, q, kv, idx, scale, rows=None):
    rows = np.arange(q.shape[0]) if rows is None else rows
    D = q.shape[2]
    kvmax = np.abs(_f(kv)).max()
    qf = _f(q[rows])
    es = D * U * scale * np.abs(qf).sum(axis=2) * kvmax  # [R, H]
    K = idx.shape[1]
    tol = 2.0 ** -8 * np.abs(want) + ((4 * es + 16 * U + K * U + 2.0 ** -8) * kvmax)[:, :, None] + 1e-30
    err = np.abs(got - want)
    bad = np.argwhere(err > tol)
    assert len(bad) == 0, f"{len(bad)} outputs outside the bound, first {bad[:3]}, err {err[tuple(bad[0])]}"


def small_case(seed, T, N, H, D, K, sink):
    q, kv, sk, idx = W.attn_inputs(seed, T, N, H, D, K, sink=sink, causal=False)
    rng = np.random.default_rng(seed)
    idx[rng.random(idx.shape) < 0.2] = -1  # holes in the lists
    idx[0, :min(4, K)] = [7, 7, 7, 3][:K]  # repeated keys
    idx[1, :] = -1  # no key
    if K > 2:
        idx[2, :] = -1
        idx[2, K - 1] = N - 1  # one key, at the end of the list
    return q, kv, sk, idx


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("H,K,sink", [(20, 77, True), (3, 32, False), (16, 1, True)])
def test_matches_oracle(dsa, D, H, K, sink):
    q, kv, sk, idx = small_case(D + H + K, 29, 300, H, D, K, sink)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(dsa, q, kv, sk, idx, scale)
    want = O.sparse_attn(q, kv, sk, idx, scale)
    check(got, want, q, kv, idx, scale)


def test_empty_lists_and_wide_logits(dsa):
    """Rows without keys give zeros (with and without a sink); logits spread over hundreds (the
    running maximum keeps e^x finite); a large sink dominates the denominator."""
    D = 64
    q, kv, _, idx = small_case(3, 9, 50, 4, D, 40, False)
    q = W.bf16_bits(_f(q) * 8.0)
    sink = np.array([0.0, 50.0, -50.0, 5.0], np.float32)
    for sk in (None, sink):
        got = run_gpu(dsa, q, kv, sk, idx, 1.0)
        want = O.sparse_attn(q, kv, sk, idx, 1.0)
        assert np.all(got[1] == 0.0)
        check(got, want, q, kv, idx, 1.0)
    empty = np.zeros((9, 0), np.int32)
    assert np.all(run_gpu(dsa, q, kv, sink, empty, 1.0) == 0.0)


@pytest.mark.parametrize("D,H", [(128, 64), (256, 40), (512, 64)])
def test_several_blocks_ragged_tail(dsa, D, H):
    """Lists of 300 entries (three 128-entry blocks, the last one partial) with holes, -1 tails
    of different lengths per row, and more rows than SMs (each CTA walks several rows)."""
    T, N, K = 200, 1000, 300
    q, kv, sk, idx = W.attn_inputs(D + H, T, N, H, D, K, causal=False)
    rng = np.random.default_rng(D)
    idx[rng.random(idx.shape) < 0.1] = -1
    for t in range(T):
        idx[t, K - (t % 150):] = -1
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(dsa, q, kv, sk, idx, scale)
    want = O.sparse_attn(q, kv, sk, idx, scale)
    check(got, want, q, kv, idx, scale)


def test_running_maximum_raised_across_blocks(dsa):
    """Scores that grow along the list (key rows scaled up with their index, wide logits): the
    running maximum is raised in later blocks, so the accumulated output and partial sums of
    earlier blocks are rescaled; with and without a sink."""
    T, N, H, D, K = 6, 640, 16, 128, 512
    q, kv, sk, idx = W.attn_inputs(41, T, N, H, D, K, causal=False)
    grow = 0.1 + 4.0 * np.arange(N) / N
    kv = W.bf16_bits(_f(kv) * grow[:, None])
    q = W.bf16_bits(_f(q) * 4.0)
    idx = np.sort(idx, axis=1)
    idx[:, :3] = -1
    for sink in (None, sk):
        got = run_gpu(dsa, q, kv, sink, idx, 1.0)
        want = O.sparse_attn(q, kv, sink, idx, 1.0)
        check(got, want, q, kv, idx, 1.0)


def test_full_size_sampled_rows(dsa):
    """The 8192-token, 64-head, D = 512 shape with causal top-2048 lists: rows sampled across the
    sequence (few keys at the start, full lists later) against the oracle."""
    T = N = 8192
    H, D, K = 64, 512, 2048
    q, kv, sk, idx = W.attn_inputs(6, T, N, H, D, K)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(dsa, q, kv, sk, idx, scale)
    rows = np.array([0, 1, 5, 100, 2047, 2048, 4000, 6001, 8191])
    want = O.sparse_attn(q[rows], kv, sk, idx[rows], scale)
    check(got[rows], want, q, kv, idx, scale, rows=rows)


@pytest.mark.parametrize("D,H,sink", [(128, 65, True), (256, 150, False), (512, 128, True)])
def test_more_than_64_heads(dsa, D, H, sink):
    """More heads than one tensor-core launch takes (64): the layer runs as head groups over the
    same lists (65 = 64 + 1, 150 = 64 + 64 + 22, 128 = 2 x 64), each group with its own sinks and
    writing its heads' slice of every output row."""
    T, N, K = 40, 600, 300
    q, kv, sk, idx = W.attn_inputs(90 + H, T, N, H, D, K, sink=sink, causal=False)
    rng = np.random.default_rng(H)
    idx[rng.random(idx.shape) < 0.1] = -1
    idx[1, :] = -1
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(dsa, q, kv, sk, idx, scale)
    want = O.sparse_attn(q, kv, sk, idx, scale)
    check(got, want, q, kv, idx, scale)


def test_128_heads_full_size_sampled_rows(dsa):
    """The 128-head shape the benchmark also times: 8192 tokens, D = 512, causal top-2048 lists
    (two head groups of 64 over 16-block lists), with a sink: rows sampled across the sequence
    against the oracle."""
    T = N = 8192
    H, D, K = 128, 512, 2048
    q, kv, sk, idx = W.attn_inputs(7, T, N, H, D, K)
    scale = 1.0 / np.sqrt(D)
    got = run_gpu(dsa, q, kv, sk, idx, scale)
    rows = np.array([0, 3, 700, 2047, 2048, 4097, 6001, 8191])
    want = O.sparse_attn(q[rows], kv, sk, idx[rows], scale)
    check(got[rows], want, q, kv, idx, scale, rows=rows)
