"""dsa_index_topk_noalloc: the fused scorer + top-k for callers that cannot allocate device memory.

Code that runs inside a memory pool or arena owning the whole device, code on a path where an
allocation would synchronise the device or fail under a hard memory cap, and runtimes that forbid
allocation after start-up cannot hand dsa_index_topk a workspace.  The allocation-free entry point
keeps that scratch in a fixed 32 MiB array inside the library.  These tests call it through the C
ABI, twice in a row on different problems (the second call finds the first call's scratch
contents), and require exactly the indices dsa_index_topk returns for the same inputs.

This file is named to be collected last, so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

DSA_ERR_WORKSPACE = 3
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def noalloc(dsa):
    lib = ctypes.CDLL(dsa.library_path())
    fn = lib.dsa_index_topk_noalloc
    p, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [p, p, p, p, p, p, i, i, i, i, i, p, p]
    fn.restype = i
    return fn


def call_noalloc(fn, t, wl, idx):
    import torch

    stream = torch.cuda.current_stream().cuda_stream
    return fn(t["q"].data_ptr(), t["w"].data_ptr(), t["k"].data_ptr(), t["k_scale"].data_ptr(),
              t["ks"].data_ptr(), t["ke"].data_ptr(), wl.T, wl.N, wl.H, wl.D, wl.topk, idx.data_ptr(), stream)


def test_noalloc_matches_dsa_index_topk_on_two_calls_in_a_row(dsa, noalloc):
    import torch

    first = W.make_config("glm")
    second = W.make_decode(seed=31, requests=64, lo=500, hi=12000, topk=256)  # rows merged from chunks
    for wl in (first, second):
        assert dsa.index_topk_workspace_size(wl.T, wl.N, wl.H, wl.D, wl.topk) <= SCRATCH_BYTES
    results = []
    for wl in (first, second):
        t = to_dev(wl)
        idx = torch.full((wl.T, wl.topk), 7, dtype=torch.int32, device="cuda")
        assert call_noalloc(noalloc, t, wl, idx) == 0
        assert dsa.get_device_error() == 0
        results.append((wl, t, idx.cpu().numpy()))
    for wl, t, got in results:
        want = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk).cpu().numpy()
        assert dsa.get_device_error() == 0
        assert np.array_equal(got, want), wl.name


def test_noalloc_few_heads_in_row_slabs(dsa, noalloc):
    """A few-head long prefill takes the routed path (scorer + selector over slabs of rows whose
    logits fit the scratch: five slabs here); the indices equal dsa_index_topk's."""
    import torch

    T = N = 6144
    ks, ke = W.causal_windows(T)
    wl = W.make_normal("fewheads", T, N, 8, 64, 512, 61, ks, ke)
    # the routed call's own workspace (a 144 MiB logits slab) exceeds the scratch: this entry
    # point accepts it all the same and runs it in slabs of floor(32 MiB / (4 N)) = 1365 rows
    assert dsa.index_topk_workspace_size(T, N, 8, 64, 512) == T * N * 4 > SCRATCH_BYTES
    t = to_dev(wl)
    idx = torch.full((wl.T, wl.topk), 7, dtype=torch.int32, device="cuda")
    assert call_noalloc(noalloc, t, wl, idx) == 0
    assert dsa.get_device_error() == 0
    want = dsa.index_topk(t["q"], t["w"], t["k"], t["k_scale"], t["ks"], t["ke"], wl.topk)
    assert dsa.get_device_error() == 0
    assert np.array_equal(idx.cpu().numpy(), want.cpu().numpy())


def test_noalloc_rejects_problems_larger_than_its_scratch(dsa, noalloc):
    import torch

    # a packed decode batch whose plan needs more than the fixed scratch: refused, nothing launched
    T, N, H, D, topk = 64, 2_000_000, 64, 128, 2048
    assert dsa.index_topk_workspace_size(T, N, H, D, topk) > SCRATCH_BYTES
    small = {"q": torch.zeros((T, H, D), dtype=torch.uint8, device="cuda"),
             "w": torch.zeros((T, H), dtype=torch.float32, device="cuda"),
             "k": torch.zeros((16, D), dtype=torch.uint8, device="cuda"),
             "k_scale": torch.zeros(16, dtype=torch.float32, device="cuda"),
             "ks": torch.zeros(T, dtype=torch.int32, device="cuda"),
             "ke": torch.zeros(T, dtype=torch.int32, device="cuda")}

    class Shape:
        pass

    wl = Shape()
    wl.T, wl.N, wl.H, wl.D, wl.topk = T, N, H, D, topk
    idx = torch.zeros((T, topk), dtype=torch.int32, device="cuda")
    assert call_noalloc(noalloc, small, wl, idx) == DSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(idx.abs().sum().item()) == 0  # untouched
