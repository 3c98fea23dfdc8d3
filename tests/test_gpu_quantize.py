"""dsa_quantize_k (e4m3 quantise-on-write of key rows) against the oracle: codes and scales
bit-exact, on random rows of many magnitudes, rows whose values sit exactly on e4m3 midpoints
(ties to even), saturating rows, zero rows and short grids, every bf16 value under many row
maxima, and the benchmark's key-cache size; then quantised keys through the fused indexer."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import overlap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_indexer_e4m3_gb300 as m
    from sparse_attention_indexer_e4m3_gb300 import build

    build.build()
    m.load()
    return m


def gpu_quantize(dsa, bits):
    import torch

    k = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)
    codes, scale = dsa.quantize_k(k)
    assert dsa.get_device_error() == 0
    return codes.cpu().numpy(), scale.cpu().numpy()


def bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def tie_rows(D, rng):
    """Rows whose largest magnitude is 448 (scale exactly 1) and whose other values are e4m3
    midpoints or values next to them (all exact in bf16)."""
    t = O.e4m3_table()[0:0x7F]
    mids = (t[:-1] + t[1:]) / 2
    mids = mids[mids < 448]
    rows = []
    for _ in range(8):
        v = rng.choice(mids, D - 1) * rng.choice([-1.0, 1.0], D - 1)
        rows.append(np.concatenate([[448.0], v]))
    return np.array(rows, np.float32)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [1, 31, 1000, 4099])
def test_codes_and_scales_bit_exact(dsa, N, D):
    rng = np.random.default_rng(N * 7 + D)
    x = rng.standard_normal((N, D)) * (10.0 ** rng.uniform(-8, 8, N))[:, None]
    bits = bf16_bits(x)
    if N > 10:
        bits[3] = 0                           # zero row
        bits[4] = 0x8000                      # -0 row
        bits[5, :] = bf16_bits(np.float32(3.0e38))[()]  # every value equal and huge
        bits[6, 1:] = 0                       # one non-zero value
    codes, scale = gpu_quantize(dsa, bits)
    c_ref, s_ref = O.quantize_rows(bits)
    assert np.array_equal(scale.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(codes, c_ref), int(np.sum(codes != c_ref))


@pytest.mark.parametrize("D", [64, 128])
def test_ties_go_to_even(dsa, D):
    rng = np.random.default_rng(D)
    x = tie_rows(D, rng)
    bits = bf16_bits(x)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), x)  # exact in bf16
    codes, scale = gpu_quantize(dsa, bits)
    c_ref, s_ref = O.quantize_rows(bits)
    assert np.all(scale == 1.0) and np.array_equal(s_ref, scale)
    assert np.array_equal(codes, c_ref)


def test_every_bf16_value_under_many_row_maxima(dsa):
    """Every finite bf16 magnitude up to the row maximum, both signs, under ~40 row maxima from
    bf16 subnormals to 3e38 (so x / s takes every kind of value: far below the e4m3 normal range,
    near its midpoints, near 448): codes and scales bit-exact.  The kernel forms most quotients
    as products with an approximate reciprocal and divides only near e4m3 midpoints, below the
    e4m3 normal range or when s has no finite reciprocal; this checks that choice exhaustively."""
    D = 128
    allbits = np.arange(0, 0x7F80, dtype=np.uint32)  # every finite non-negative bf16 pattern
    rng = np.random.default_rng(11)
    maxima = np.concatenate([[0x0001, 0x0003, 0x007F, 0x0080, 0x0081, 0x3F80, 0x43E0, 0x7F7F],
                             rng.integers(0x0100, 0x7F7F, 32)]).astype(np.uint32)
    rows = []
    for mb in maxima:
        xs = allbits[allbits <= mb]
        xs = np.concatenate([xs, xs | 0x8000])
        pad = (-len(xs)) % (D - 1)
        xs = np.concatenate([xs, np.zeros(pad, np.uint32)]).reshape(-1, D - 1)
        rows.append(np.concatenate([np.full((len(xs), 1), mb, np.uint32), xs], axis=1))
    bits = np.concatenate(rows).astype(np.uint16)
    codes, scale = gpu_quantize(dsa, bits)
    c_ref, s_ref = O.quantize_rows(bits)
    assert np.array_equal(scale.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(codes, c_ref), int(np.sum(codes != c_ref))


def test_key_cache_of_the_benchmark_size_sampled_rows(dsa):
    """The shape the benchmark times: 1,939,851 rows of D = 128 seeded normal bf16 keys in one
    launch; every 97th row (and the last) against the oracle, bit-exact."""
    N, D = 1_939_851, 128
    bits = W.bf16_bits(W.normal(17, 21, N * D)).reshape(N, D)
    codes, scale = gpu_quantize(dsa, bits)
    rows = np.concatenate([np.arange(0, N, 97), [N - 1]])
    c_ref, s_ref = O.quantize_rows(bits[rows])
    assert np.array_equal(scale[rows].view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(codes[rows], c_ref), int(np.sum(codes[rows] != c_ref))


def test_quantised_keys_through_the_indexer(dsa):
    """Keys quantised on the GPU feed dsa_index_topk; the oracle scores the oracle-quantised keys
    (the same codes and scales) and its top-k matches."""
    import torch

    rng = np.random.default_rng(5)
    T, N, H, D, topk = 64, 3000, 32, 128, 256
    kf = rng.standard_normal((N, D)).astype(np.float32) * (1 + 3 * (rng.random((N, 1)) < 0.01))
    bits = bf16_bits(kf)
    codes, scale = gpu_quantize(dsa, bits)
    c_ref, s_ref = O.quantize_rows(bits)
    assert np.array_equal(codes, c_ref) and np.array_equal(scale, s_ref)
    ks = np.zeros(T, np.int32)
    ke = np.full(T, N, np.int32)
    wl = W.make_normal("qk", T, N, H, D, topk, 9, ks, ke)
    d = {n: torch.from_numpy(np.ascontiguousarray(getattr(wl, n))).cuda() for n in ("q", "w", "ks", "ke")}
    kc = torch.from_numpy(codes).cuda()
    kscale = torch.from_numpy(scale).cuda()
    idx = dsa.index_topk(d["q"], d["w"], kc, kscale, d["ks"], d["ke"], topk).cpu().numpy()
    assert dsa.get_device_error() == 0
    ref = O.index_score(wl.q, wl.w, c_ref, s_ref, ks, ke)
    assert overlap(idx, O.topk(ref, topk)) >= 0.999
