"""dsa_sparse_attn_bwd (and the forward's lse output) against the oracle's gradients.

The GPU rounds the softmax weights P and the score gradients dS to bf16 before the products that
use them (as the forward rounds its weights), takes delta from the forward's bf16 output, and
accumulates in fp32.  Per gradient entry the error is therefore bounded by a small multiple of
2^-8 times the sum of the magnitudes of the terms that make it up:
  * dS_j = scale p_j (dP_j - delta): p_j and the product carry 2^-9 relative from the bf16
    rounding; delta carries 2^-9 of D_lt = sum_d |o_d| |do_d| from the bf16 output; so
    |err(dS_j)| <= 2^-8 scale p_j (|dP_j| + |delta| + D_lt);
  * dq[t,h,d] = sum_j dS_j kv[j,d]       -> R_dq = scale sum_j p_j (|dP_j| + |delta| + D_lt) |kv[j,d]|
  * dkv[j,d] += dS_j q[t,h,d] + p_j do[t,h,d]
                                         -> R_dkv = sum over listings of
                                            scale p_j (|dP_j| + |delta| + D_lt) |q[t,h,d]| + p_j |do[t,h,d]|
  * dsink[h] = -sum_t p_sink delta       -> R_sink = sum_t p_sink (|delta| + D_lt)
and the test allows 2^-7 R + 1e-6 (twice the estimate; the fp32 sums add far less).
lse: |lse_gpu - lse| <= 2^-20 (|lse| + 1) (fp32 sums of exponentials).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def _f(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf(t):
    import torch

    return torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).cuda().view(torch.bfloat16)


def run_gpu(dsa, q, kv, sink, idx, do, scale):
    import torch

    qt, kvt, dot = _bf(q), _bf(kv), _bf(do)
    it = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    st = None if sink is None else torch.from_numpy(sink).cuda()
    T, H, D = q.shape
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    out = dsa.sparse_attn(qt, kvt, it, attn_sink=st, scale=scale, lse=lse)
    dq, dkv, dsink = dsa.sparse_attn_bwd(qt, kvt, it, out, lse, dot, attn_sink=st, scale=scale)
    assert dsa.get_device_error() == 0
    return (lse.cpu().numpy().astype(np.float64), dq.cpu().numpy().astype(np.float64),
            dkv.cpu().numpy().astype(np.float64), None if dsink is None else dsink.cpu().numpy().astype(np.float64))


def reference_terms(q, kv, sink, idx, do, scale):
    """Per (row, head): the exact lse, and the magnitude sums R_dq, R_dkv, R_sink of the module
    docstring (numpy, double)."""
    qf, kvf, dof = _f(q), _f(kv), _f(do)
    T, H, D = qf.shape
    N = kvf.shape[0]
    lse = np.full((T, H), -np.inf)
    r_dq = np.zeros((T, H, D))
    r_dkv = np.zeros((N, D))
    r_sink = np.zeros(H)
    for t in range(T):
        lst = idx[t][(idx[t] >= 0) & (idx[t] < N)]
        if len(lst) == 0:
            if sink is not None:
                lse[t] = sink.astype(np.float64)
            continue
        v = kvf[lst]                           # [L, D]
        s = scale * (qf[t] @ v.T)              # [H, L]
        if sink is not None:
            m = np.maximum(s.max(axis=1), sink.astype(np.float64))
            z = np.exp(s - m[:, None]).sum(axis=1) + np.exp(sink.astype(np.float64) - m)
        else:
            m = s.max(axis=1)
            z = np.exp(s - m[:, None]).sum(axis=1)
        lse[t] = m + np.log(z)
        p = np.exp(s - lse[t][:, None])        # [H, L]
        o = p @ v                              # [H, D]
        dp = dof[t] @ v.T                      # [H, L]
        delta = (dof[t] * o).sum(axis=1)       # [H]
        dlt = (np.abs(dof[t]) * np.abs(o)).sum(axis=1)
        w = scale * p * (np.abs(dp) + np.abs(delta)[:, None] + dlt[:, None])  # [H, L]
        r_dq[t] = w @ np.abs(v)
        contrib = w.T @ np.abs(qf[t]) + p.T @ np.abs(dof[t])  # [L, D]
        np.add.at(r_dkv, lst, contrib)
        if sink is not None:
            r_sink += np.exp(sink.astype(np.float64) - lse[t]) * (np.abs(delta) + dlt)
    return lse, r_dq, r_dkv, r_sink


def sanitized(idx, N):
    """The lists as the oracle takes them: an entry outside [0, N), which the kernels skip like
    -1, is written as -1 (the oracle rejects it)."""
    return np.where((idx < 0) | (idx >= N), -1, idx).astype(np.int32)


def check(dsa, q, kv, sink, idx, do, scale):
    lse_g, dq_g, dkv_g, ds_g = run_gpu(dsa, q, kv, sink, idx, do, scale)
    dq_o, dkv_o, ds_o = O.sparse_attn_bwd(q, kv, sink, sanitized(idx, kv.shape[0]), do, scale)
    lse_r, r_dq, r_dkv, r_sink = reference_terms(q, kv, sink, idx, do, scale)
    fin = np.isfinite(lse_r)
    assert np.array_equal(np.isfinite(lse_g), fin)
    assert np.all(np.abs(lse_g[fin] - lse_r[fin]) <= 2.0 ** -20 * (np.abs(lse_r[fin]) + 1.0))
    tol = 2.0 ** -7
    assert np.all(np.abs(dq_g - dq_o) <= tol * r_dq + 1e-6), np.max(np.abs(dq_g - dq_o) / (tol * r_dq + 1e-6))
    assert np.all(np.abs(dkv_g - dkv_o) <= tol * r_dkv + 1e-6), np.max(np.abs(dkv_g - dkv_o) / (tol * r_dkv + 1e-6))
    if sink is None:
        assert ds_g is None
    else:
        assert np.all(np.abs(ds_g - ds_o) <= tol * r_sink + 1e-6)


def lists(seed, T, N, K):
    """Selector-like causal lists plus the edge cases: -1 holes, a repeated key, a row without
    keys, entries out of [0, N) (skipped like -1), a row whose only key sits in its last block."""
    idx = W.attn_indices(seed, T, N, K, causal=True)
    rng = np.random.default_rng(seed)
    holes = rng.random(idx.shape) < 0.1
    idx[holes] = -1
    idx[1, :4] = [5, 5, 5, 9]
    idx[2, :] = -1
    idx[3, 0] = N + 3
    idx[3, 1] = -7
    idx[4, :] = -1
    idx[4, K - 1] = 0
    return idx


@pytest.mark.parametrize("D,H,sink", [(128, 64, True), (128, 64, False), (256, 40, True), (128, 16, False),
                                      (256, 64, False)])
def test_several_blocks_ragged_tail(dsa, D, H, sink):
    T, N, K = 48, 700, 300  # three 128-entry blocks per full row, the last one partial
    q, kv, sk, _ = W.attn_inputs(51 + D + H, T, N, H, D, K, sink=sink)
    idx = lists(52 + H, T, N, K)
    do = W.bf16_bits(W.normal(53 + H, 13, T * H * D)).reshape(T, H, D)
    check(dsa, q, kv, sk, idx, do, 1.0 / np.sqrt(D))


@pytest.mark.parametrize("D,H,sink", [(128, 65, True), (256, 128, True), (128, 150, False)])
def test_more_than_64_heads(dsa, D, H, sink):
    """More heads than one launch takes (64): head groups over the same lists (65 = 64 + 1,
    128 = 2 x 64, 150 = 64 + 64 + 22), every group adding into the one dkv; lse, dq and dsink
    at each head's own position."""
    T, N, K = 24, 500, 260
    q, kv, sk, _ = W.attn_inputs(91 + H, T, N, H, D, K, sink=sink)
    idx = lists(92 + H, T, N, K)
    do = W.bf16_bits(W.normal(93 + H, 13, T * H * D)).reshape(T, H, D)
    check(dsa, q, kv, sk, idx, do, 1.0 / np.sqrt(D))


def test_many_rows_share_keys(dsa):
    """More rows than SMs and heavily shared keys, so the atomic sums into dkv meet from many
    CTAs at once."""
    T, N, K, H, D = 400, 160, 128, 64, 128
    q, kv, sk, idx = W.attn_inputs(61, T, N, H, D, K, sink=True, causal=False)
    do = W.bf16_bits(W.normal(62, 13, T * H * D)).reshape(T, H, D)
    check(dsa, q, kv, sk, idx, do, 0.1)


def test_mid_size_full_parity(dsa):
    """512 rows of top-384 causal lists over 1024 keys, 64 heads, D = 128, with a sink: every
    gradient entry against the oracle."""
    T, N, K, H, D = 512, 1024, 384, 64, 128
    q, kv, sk, idx = W.attn_inputs(65, T, N, H, D, K, sink=True)
    do = W.bf16_bits(W.normal(66, 13, T * H * D)).reshape(T, H, D)
    check(dsa, q, kv, sk, idx, do, 1.0 / np.sqrt(D))


def test_large_prefill_sampled_rows(dsa):
    """A 4096-token, 64-head, D = 128 prefill over top-2048 causal lists (16 blocks per full row):
    dq and lse on sampled rows against the oracle (a row's dq depends on that row alone)."""
    T, N, K, H, D = 4096, 4096, 2048, 64, 128
    q, kv, _, idx = W.attn_inputs(71, T, N, H, D, K, sink=False)
    do = W.bf16_bits(W.normal(72, 13, T * H * D)).reshape(T, H, D)
    scale = 1.0 / np.sqrt(D)
    lse_g, dq_g, dkv_g, _ = run_gpu(dsa, q, kv, None, idx, do, scale)
    rows = np.concatenate([np.arange(0, T, 256), [1, 2047, 2048, T - 1]])
    dq_o, _, _ = O.sparse_attn_bwd(q[rows], kv, None, idx[rows], do[rows], scale)
    lse_r, r_dq, _, _ = reference_terms(q[rows], kv, None, idx[rows], do[rows], scale)
    assert np.all(np.abs(dq_g[rows] - dq_o) <= 2.0 ** -7 * r_dq + 1e-6)
    assert np.all(np.abs(lse_g[rows] - lse_r) <= 2.0 ** -20 * (np.abs(lse_r) + 1.0))
    assert np.all(np.isfinite(dkv_g))


def test_bench_shape_sampled_rows(dsa):
    """The shape the benchmark times: 8192 rows of causal top-2048 lists over 8192 keys, 64 heads,
    D = 256, with a sink: dq and lse on sampled rows against the oracle, dsink and dkv finite."""
    T, N, K, H, D = 8192, 8192, 2048, 64, 256
    q, kv, sk, idx = W.attn_inputs(81, T, N, H, D, K, sink=True)
    do = W.bf16_bits(W.normal(82, 13, T * H * D)).reshape(T, H, D)
    scale = 1.0 / np.sqrt(D)
    lse_g, dq_g, dkv_g, ds_g = run_gpu(dsa, q, kv, sk, idx, do, scale)
    rows = np.concatenate([np.arange(0, T, 512), [1, 2047, 2048, 4097, T - 1]])
    dq_o, _, _ = O.sparse_attn_bwd(q[rows], kv, sk, idx[rows], do[rows], scale)
    lse_r, r_dq, _, _ = reference_terms(q[rows], kv, sk, idx[rows], do[rows], scale)
    assert np.all(np.abs(dq_g[rows] - dq_o) <= 2.0 ** -7 * r_dq + 1e-6)
    assert np.all(np.abs(lse_g[rows] - lse_r) <= 2.0 ** -20 * (np.abs(lse_r) + 1.0))
    assert np.all(np.isfinite(dkv_g)) and np.all(np.isfinite(ds_g))


def test_argument_errors(dsa):
    import torch

    T, N, K, H, D = 4, 16, 8, 4, 64
    z = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((N, D), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    lse = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    with pytest.raises(dsa.DsaError, match="UNSUPPORTED"):  # D = 64 has no backward kernel
        dsa.sparse_attn_bwd(z, kv, idx, z, lse, z)
    z2 = torch.zeros((T, H, 512), dtype=torch.bfloat16, device="cuda")
    kv2 = torch.zeros((N, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError, match="UNSUPPORTED"):  # nor D = 512
        dsa.sparse_attn_bwd(z2, kv2, idx, z2, lse, z2)
    assert dsa.get_device_error() == 0
