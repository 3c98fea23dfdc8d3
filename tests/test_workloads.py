"""The seeded input generators (host logic, CPU): determinism and the structure the parity
tests and the bench rely on."""
import numpy as np

import workloads as W


def test_bf16_rounding_matches_torch():
    import torch

    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4096) * 10.0 ** rng.integers(-30, 30, 4096),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, -2.5, 3.0e38, 1e-40]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.bf16_bits(x), want)
    # random finite float32 bit patterns, and exact halfway cases (low 16 bits 0x8000) on both
    # parities of the kept bits, up to the largest finite values
    bits = rng.integers(0, 2 ** 32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, 4096, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    f = np.concatenate([bits, ties, np.array([0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0x00008000], np.uint32)]).view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = W.bf16_bits(f.astype(np.float64))
    ok = np.isfinite((want.astype(np.uint32) << 16).view(np.float32))  # (values that round past the
    assert np.array_equal(got[ok], want[ok])                           # largest bf16 are not inputs)


def test_attention_index_lists():
    T, N, K = 300, 250, 64
    idx = W.attn_indices(4, T, N, K)
    assert idx.shape == (T, K) and idx.dtype == np.int32
    for t in range(T):
        n = min(t + 1, N)
        row = idx[t]
        m = min(K, n)
        assert np.all(row[m:] == -1)
        sel = row[:m]
        assert np.all(sel >= 0) and np.all(sel < n)  # causal
        assert np.all(np.diff(sel) > 0)  # ascending, distinct
    assert np.array_equal(idx, W.attn_indices(4, T, N, K))  # a pure function of the seed
    assert not np.array_equal(idx, W.attn_indices(5, T, N, K))
    full = W.attn_indices(4, 3, 10, 8, causal=False)
    assert np.all(full >= 0)


def test_attention_inputs_shapes_and_determinism():
    q, kv, sink, idx = W.attn_inputs(2, 17, 40, 3, 64, 9)
    assert q.shape == (17, 3, 64) and q.dtype == np.uint16
    assert kv.shape == (40, 64) and kv.dtype == np.uint16
    assert sink.shape == (3,) and sink.dtype == np.float32
    assert idx.shape == (17, 9)
    q2, kv2, sink2, idx2 = W.attn_inputs(2, 17, 40, 3, 64, 9)
    assert np.array_equal(q, q2) and np.array_equal(kv, kv2) and np.array_equal(sink, sink2)
    assert np.array_equal(idx, idx2)
    assert W.attn_inputs(2, 17, 40, 3, 64, 9, sink=False)[2] is None
