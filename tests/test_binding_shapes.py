"""Host logic of the Python binding (CPU): every entry point accepts correctly shaped tensors and
rejects a caller buffer of the wrong shape before anything reaches the library.  The library is
replaced by a stub and CPU tensors stand in for device ones, so no GPU is involved."""
import pytest
import torch

import sparse_attention_indexer_e4m3_gb300 as dsa

T, N, H, D, K = 6, 40, 4, 64, 5


@pytest.fixture()
def stub(monkeypatch):
    calls = []

    class Lib:
        def __getattr__(self, name):
            def fn(*args):
                calls.append(name)
                return 0
            return fn

    def dev(t, name, dtypes):
        if t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        assert t.dtype in dtypes, name
        return t

    real_empty = torch.empty
    monkeypatch.setattr(dsa, "load", lambda: Lib())
    monkeypatch.setattr(dsa, "_dev", dev)
    monkeypatch.setattr(dsa, "_stream_ptr", lambda s: 0)
    monkeypatch.setattr(dsa, "_workspace", lambda need, ws, device: (None, 0))
    monkeypatch.setattr(torch, "empty", lambda *a, **kw: real_empty(*a, **{k: v for k, v in kw.items() if k != "device"}))
    return calls


def _indexer_inputs():
    return (torch.zeros((T, H, D), dtype=torch.uint8), torch.zeros((T, H)), torch.zeros((N, D), dtype=torch.uint8),
            torch.zeros(N), torch.zeros(T, dtype=torch.int32), torch.zeros(T, dtype=torch.int32))


def test_valid_shapes_reach_the_library(stub):
    q, w, k, ksc, ks, ke = _indexer_inputs()
    dsa.index_score(q, w, k, ksc, ks, ke)
    dsa.topk(torch.zeros((T, N)), ks, ke, K)
    dsa.index_topk(q, w, k, ksc, ks, ke, K)
    dsa.index_topk_plan(ks, ke, N, H, D, K)
    dsa.index_topk_run(q, w, k, ksc, ks, ke, K, None)
    dsa.quantize_k(torch.zeros((N, D), dtype=torch.bfloat16))
    dsa.sparse_attn(torch.zeros((T, H, D), dtype=torch.bfloat16), torch.zeros((N, D), dtype=torch.bfloat16),
                    torch.zeros((T, K), dtype=torch.int32), attn_sink=torch.zeros(H))
    for name in ("dsa_index_score", "dsa_topk", "dsa_index_topk", "dsa_index_topk_plan", "dsa_index_topk_run",
                 "dsa_quantize_k", "dsa_sparse_attn"):
        assert name in stub


def test_wrong_buffers_are_rejected(stub):
    q, w, k, ksc, ks, ke = _indexer_inputs()
    i32 = torch.int32
    bad = [
        lambda: dsa.index_score(q, w, k, ksc, ks, ke, logits=torch.zeros((T, N + 1))),
        lambda: dsa.topk(torch.zeros((T, N)), ks, ke, K, idx=torch.zeros((T, K + 1), dtype=i32)),
        lambda: dsa.topk(torch.zeros((T, N)), ks[:3], ke, K),
        lambda: dsa.index_topk(q, w, k, ksc, ks, ke, K, idx=torch.zeros((T - 1, K), dtype=i32)),
        lambda: dsa.index_topk(q, w, k, ksc, ks[:2], ke, K),
        lambda: dsa.index_topk_run(q, w, k, ksc, ks, ke, K, None, idx=torch.zeros((T, K - 1), dtype=i32)),
        lambda: dsa.index_topk_plan(ks, ke[:2], N, H, D, K),
        lambda: dsa.quantize_k(torch.zeros((N, D), dtype=torch.bfloat16), codes=torch.zeros((N, D + 1), dtype=torch.uint8)),
        lambda: dsa.quantize_k(torch.zeros((N, D), dtype=torch.bfloat16), scale=torch.zeros(N - 1)),
        lambda: dsa.sparse_attn(torch.zeros((T, H, D), dtype=torch.bfloat16), torch.zeros((N, D), dtype=torch.bfloat16),
                                torch.zeros((T, K), dtype=i32), out=torch.zeros((T, H, D - 1), dtype=torch.bfloat16)),
        lambda: dsa.sparse_attn(torch.zeros((T, H, D), dtype=torch.bfloat16), torch.zeros((N, D), dtype=torch.bfloat16),
                                torch.zeros((T, K), dtype=i32), attn_sink=torch.zeros(H + 1)),
        lambda: dsa.sparse_attn(torch.zeros((T, H, D), dtype=torch.bfloat16), torch.zeros((N, D + 2), dtype=torch.bfloat16),
                                torch.zeros((T, K), dtype=i32)),
    ]
    for i, f in enumerate(bad):
        with pytest.raises(ValueError):
            f()
    assert stub == []  # nothing reached the library
