"""Seeded synthetic inputs for the FP8 lightning indexer and top-k selector.

This package makes inputs only.  It holds none of the indexer's arithmetic, so the CPU
oracle and the CUDA path can both consume it without sharing any of the method.  The
random numbers come from ``gen.c`` (counter-based SplitMix64 + Box-Muller), so every
byte is a pure function of (seed, stream, index) and is identical on every machine.

The five recipes follow the workloads described for the DeepSeek-V3.2 lightning indexer
(TileLang ``examples/deepseek_v32`` README, "Lightning Indexer" and "Top-k Selector")
and the SM100 prefill scorer page (Modular ``sparse_index_fp8_sm100_prefill``, the
GLM and 64-head prefill shapes):

===========  =====================================================================
name         recipe
===========  =====================================================================
tiny         T=N=256, H=4, D=64, causal (ks=0, ke=t+1), top-k 32, seed 0
glm          T=N=1024, H=32, D=128, causal, top-k 512, seed 1
dsv32        T=N=8192, H=64, D=128, causal, top-k 2048, seed 2
decode       64 requests x 1 token, cache lengths uniform in [4096, 65536] packed
             along N with ks/ke = request offsets, H=64, D=128, top-k 2048, seed 3
varlen       documents 2048/6144/8192/16384 packed to T=N=32768, ks=doc start,
             ke=t+1, 1% of keys (chosen uniformly) scaled x8 before quantisation,
             H=64, D=128, top-k 2048, seed 4
===========  =====================================================================

Value recipe (all configs): q[t,h,:] and k[j,:] are N(0,1) draws quantised per row to
e4m3 with scale max|row|/448; k_scale[j] is that key's scale; w[t,h] ~ N(0, std 1/sqrt(H))
is multiplied by the q row's scale (the q dequantisation folded into the head weight),
then stored as fp32.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libwlgen.so")
_lib = None
_lib_lock = threading.Lock()

# stream ids (one independent random stream per input tensor)
STREAM_Q = 1
STREAM_K = 2
STREAM_W = 3
STREAM_LEN = 4
STREAM_HEAVY = 5
STREAM_INT_Q = 11
STREAM_INT_K = 12
STREAM_INT_W = 13
STREAM_INT_KS = 14


def build(force: bool = False) -> str:
    """Compile gen.c into libwlgen.so next to it (plain gcc, no architecture flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
            p = ctypes.c_void_p
            lib.wl_u64.restype = u64
            lib.wl_u64.argtypes = [u64, u64, u64]
            lib.wl_e4m3_encode.restype = ctypes.c_uint8
            lib.wl_e4m3_encode.argtypes = [ctypes.c_double]
            lib.wl_normal.argtypes = [u64, u64, i64, ctypes.c_double, p, i32]
            lib.wl_uniform.argtypes = [u64, u64, i64, p]
            lib.wl_uniform_int.argtypes = [u64, u64, i64, i64, i64, p]
            lib.wl_normal_e4m3_rows.argtypes = [u64, u64, i64, i64, p, p, p, i32]
            lib.wl_encode_e4m3.argtypes = [p, i64, p]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, stream: int, n: int, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().wl_normal(seed, stream, n, std, _ptr(out), _threads())
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().wl_uniform(seed, stream, n, _ptr(out))
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    _load().wl_uniform_int(seed, stream, n, lo, hi, _ptr(out))
    return out


def encode_e4m3(values) -> np.ndarray:
    """Round-to-nearest-even saturating e4m3 codes of float64 values (input preparation)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().wl_encode_e4m3(_ptr(v), v.size, _ptr(out))
    return out


def normal_e4m3_rows(seed: int, stream: int, rows: int, cols: int, row_mult=None):
    """Per-row quantised N(0,1) matrix: (codes uint8 [rows, cols], scales float64 [rows])."""
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float64)
    rm = None
    if row_mult is not None:
        rm = np.ascontiguousarray(row_mult, dtype=np.float64)
        assert rm.shape == (rows,)
    _load().wl_normal_e4m3_rows(seed, stream, rows, cols, None if rm is None else _ptr(rm), _ptr(codes),
                                _ptr(scales), _threads())
    return codes, scales


@dataclass
class Workload:
    """One indexer problem.  Layouts are those of the C-ABI: row-major, contiguous."""

    name: str
    T: int
    N: int
    H: int
    D: int
    topk: int
    q: np.ndarray  # uint8 e4m3 codes [T, H, D]
    w: np.ndarray  # float32 [T, H]
    k: np.ndarray  # uint8 e4m3 codes [N, D]
    k_scale: np.ndarray  # float32 [N]
    ks: np.ndarray  # int32 [T]
    ke: np.ndarray  # int32 [T]
    meta: dict = field(default_factory=dict)

    @property
    def pairs(self) -> int:
        lo = np.clip(self.ks.astype(np.int64), 0, self.N)
        hi = np.clip(self.ke.astype(np.int64), 0, self.N)
        return int(np.maximum(hi - lo, 0).sum())


def causal_windows(T: int, doc_lens=None):
    """ks = start of the token's document, ke = t + 1 (inclusive causal window)."""
    ks = np.zeros(T, dtype=np.int32)
    if doc_lens is not None:
        start = 0
        for L in doc_lens:
            ks[start:start + L] = start
            start += L
        assert start == T
    ke = np.arange(1, T + 1, dtype=np.int32)
    return ks, ke


def make_normal(name: str, T: int, N: int, H: int, D: int, topk: int, seed: int, ks, ke,
                heavy_frac: float = 0.0, heavy_mult: float = 8.0, meta=None) -> Workload:
    """Normal-valued e4m3 problem per the value recipe in the module docstring."""
    q_codes, q_scale = normal_e4m3_rows(seed, STREAM_Q, T * H, D)
    row_mult = None
    if heavy_frac > 0.0:
        u = uniform(seed, STREAM_HEAVY, N)
        row_mult = np.where(u < heavy_frac, heavy_mult, 1.0)
    k_codes, k_scale = normal_e4m3_rows(seed, STREAM_K, N, D, row_mult)
    w = normal(seed, STREAM_W, T * H, std=1.0 / math.sqrt(H)) * q_scale
    m = dict(meta or {})
    if row_mult is not None:
        m["heavy_keys"] = int((row_mult != 1.0).sum())
    return Workload(name=name, T=T, N=N, H=H, D=D, topk=topk,
                    q=q_codes.reshape(T, H, D), w=w.astype(np.float32).reshape(T, H),
                    k=k_codes, k_scale=k_scale.astype(np.float32),
                    ks=np.ascontiguousarray(ks, dtype=np.int32), ke=np.ascontiguousarray(ke, dtype=np.int32),
                    meta=m)


def decode_lengths(seed: int, requests: int = 64, lo: int = 4096, hi: int = 65536) -> np.ndarray:
    return uniform_int(seed, STREAM_LEN, requests, lo, hi)


def make_decode(seed: int = 3, requests: int = 64, lo: int = 4096, hi: int = 65536, H: int = 64, D: int = 128,
                topk: int = 2048, name: str = "decode") -> Workload:
    """Ragged decode: one query token per request, the request's cache packed along N."""
    lens = decode_lengths(seed, requests, lo, hi)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    N = int(lens.sum())
    ks = starts.astype(np.int32)
    ke = (starts + lens).astype(np.int32)
    return make_normal(name, requests, N, H, D, topk, seed, ks, ke, meta={"lengths": lens.tolist()})


VARLEN_DOCS = (2048, 6144, 8192, 16384)


def make_config(name: str) -> Workload:
    """The five named workloads (see the module docstring)."""
    if name == "tiny":
        ks, ke = causal_windows(256)
        return make_normal("tiny", 256, 256, 4, 64, 32, 0, ks, ke)
    if name == "glm":
        ks, ke = causal_windows(1024)
        return make_normal("glm", 1024, 1024, 32, 128, 512, 1, ks, ke)
    if name == "dsv32":
        ks, ke = causal_windows(8192)
        return make_normal("dsv32", 8192, 8192, 64, 128, 2048, 2, ks, ke)
    if name == "decode":
        return make_decode()
    if name == "varlen":
        T = sum(VARLEN_DOCS)
        ks, ke = causal_windows(T, VARLEN_DOCS)
        return make_normal("varlen", T, T, 64, 128, 2048, 4, ks, ke, heavy_frac=0.01, heavy_mult=8.0,
                           meta={"docs": list(VARLEN_DOCS)})
    raise KeyError(name)


CONFIG_NAMES = ("tiny", "glm", "dsv32", "decode", "varlen")


def make_integer(name: str, T: int, N: int, H: int, D: int, topk: int, seed: int, ks, ke) -> Workload:
    """Inputs on which every product and partial sum is exactly representable in fp32.

    q, k are integers in [-4, 4] (exact in e4m3), w in {+-0.5, +-1, +-2}, k_scale in
    {0.5, 1, 2}.  Used to check that the GPU's fp32 scores are bit-exact.
    """
    qv = uniform_int(seed, STREAM_INT_Q, T * H * D, -4, 4).astype(np.float64)
    kv = uniform_int(seed, STREAM_INT_K, N * D, -4, 4).astype(np.float64)
    wsel = uniform_int(seed, STREAM_INT_W, T * H, 0, 5)
    wvals = np.array([0.5, -0.5, 1.0, -1.0, 2.0, -2.0])[wsel]
    kssel = uniform_int(seed, STREAM_INT_KS, N, 0, 2)
    ksv = np.array([0.5, 1.0, 2.0])[kssel]
    return Workload(name=name, T=T, N=N, H=H, D=D, topk=topk,
                    q=encode_e4m3(qv).reshape(T, H, D), w=wvals.astype(np.float32).reshape(T, H),
                    k=encode_e4m3(kv).reshape(N, D), k_scale=ksv.astype(np.float32),
                    ks=np.ascontiguousarray(ks, dtype=np.int32), ke=np.ascontiguousarray(ke, dtype=np.int32))


# ------------------------------------------------------------------ sparse-attention inputs


def bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns (uint16) of float64 values: to float32, then round to nearest even on
    the upper 16 bits (input preparation; finite values only)."""
    # (in uint32: for a finite value the largest pattern, 0xFF7FFFFF, plus 0x8000 stays below 2^32)
    b = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32)
    r = (b >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def attn_indices(seed: int, T: int, N: int, K: int, causal: bool = True) -> np.ndarray:
    """int32 [T, K] index lists shaped like the selector's output: row t holds min(K, n_t)
    distinct keys drawn uniformly from its n_t = min(t + 1, N) causal keys (all N keys when not
    causal), in ascending order, then -1 padding."""
    idx = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        n = min(t + 1, N) if causal else N
        m = min(K, n)
        if m == 0:
            continue
        if m == n:
            idx[t, :m] = np.arange(n, dtype=np.int32)
        else:
            r = uniform(seed, 1000 + t, n)
            idx[t, :m] = np.sort(np.argsort(r, kind="stable")[:m]).astype(np.int32)
    return idx


def attn_inputs(seed: int, T: int, N: int, H: int, D: int, K: int, sink: bool = True, causal: bool = True):
    """(q bf16 bits [T, H, D], kv bf16 bits [N, D], attn_sink float32 [H] or None, idx [T, K]):
    q and kv N(0, 1), the sink N(0, 1) per head, idx from attn_indices."""
    q = bf16_bits(normal(seed, 10, T * H * D)).reshape(T, H, D)
    kv = bf16_bits(normal(seed, 11, N * D)).reshape(N, D)
    sk = normal(seed, 12, H).astype(np.float32) if sink else None
    return q, kv, sk, attn_indices(seed, T, N, K, causal)
