"""CPU oracle for the FP8 lightning indexer and exact top-k selector.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py``, never by the library.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.cpp`` (plain C++17, double precision, full sort); this module
compiles it with g++ and marshals numpy arrays.  What each function follows:

* ``e4m3_table`` -- OCP E4M3FN bit-field decode (TileLang deepseek_v32 README, "Lightning
  Indexer": fp8 index vectors; FlashInfer MLA-decode discussion: e4m3 max 448).
* ``index_score`` -- Modular ``sparse_index_fp8_sm100_prefill``, the per-(token, key) logit
  formula; TileLang README, "Lightning Indexer" (relu, head weight, key scale, head sum, and
  the per-token key window clamped to the key count).
* ``topk`` / ``topk_dense`` -- TileLang README, "Top-k Selector" (k largest per row within the
  window), ties to the lower key index, indices ascending, ``-1`` padding as in the DeepSeek
  V4.1 ``sparse_attn_kernel`` page.
* ``quantize_rows`` / ``e4m3_encode`` -- the fp8 index keys' quantisation (TileLang README,
  "Lightning Indexer": FP8-quantized index vectors; e4m3 max 448): per row s = max|x| / 448,
  codes = nearest e4m3 of x / s, ties to even, saturating; brute-force nearest value.
* ``sparse_attn`` -- attention over the listed keys (DeepSeek V4.1 ``sparse_attn_kernel`` page;
  TileLang README, "Sparse MLA Forward"): per head, softmax of scale * q.kv over the list's
  non-negative entries with an optional per-head sink in the denominator, weights applied to
  the same kv rows; an empty list gives 0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with g++ -O2 (IEEE semantics: no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp, src, "-lpthread"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_e4m3_table.argtypes = [p]
    lib.oracle_e4m3_table.restype = None
    lib.oracle_window_lengths.argtypes = [p, p, i64, i64, p, i64, p, p]
    lib.oracle_window_lengths.restype = i32
    lib.oracle_index_score.argtypes = [p, p, p, p, p, p, i64, i64, i32, i32, p, i64, p, p, i32]
    lib.oracle_index_score.restype = i32
    lib.oracle_topk_compact.argtypes = [p, p, p, p, i64, i32, p, i32]
    lib.oracle_topk_compact.restype = i32
    lib.oracle_quantize_rows.argtypes = [p, i64, i64, p, p]
    lib.oracle_quantize_rows.restype = i32
    lib.oracle_e4m3_encode.argtypes = [p, i64, p]
    lib.oracle_e4m3_encode.restype = i32
    lib.oracle_sparse_attn.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, ctypes.c_double, p, i32]
    lib.oracle_sparse_attn.restype = i32
    lib.oracle_sparse_attn_bwd.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, ctypes.c_double, p, p, p, i32]
    lib.oracle_sparse_attn_bwd.restype = i32
    for name in ("oracle_topk_f64", "oracle_topk_f32"):
        fn = getattr(lib, name)
        fn.argtypes = [p, i64, p, p, i64, i64, i32, p, i32]
        fn.restype = i32
    return lib


def load_library(path: str):
    """Load (and bind) an oracle shared library from an explicit path."""
    return _bind(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def threads() -> int:
    """Host threads the oracle uses (all cores of this machine)."""
    return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def e4m3_table(lib=None) -> np.ndarray:
    lib = lib or _load()
    out = np.empty(256, dtype=np.float64)
    lib.oracle_e4m3_table(_p(out))
    return out


def e4m3_encode(y, lib=None) -> np.ndarray:
    """Nearest e4m3 codes of float32 values (ties to even, saturating at 448)."""
    lib = lib or _load()
    y = _c(y, np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode(_p(y), y.size, _p(out))
    return out


def quantize_rows(x_bf16_bits, lib=None):
    """Quantise rows of bf16 values (uint16 bit patterns, [N, D]) to e4m3 codes [N, D] and
    per-row fp32 scales [N]."""
    lib = lib or _load()
    x = _c(x_bf16_bits, np.uint16)
    N, D = x.shape
    codes = np.empty((N, D), dtype=np.uint8)
    scale = np.empty(N, dtype=np.float32)
    lib.oracle_quantize_rows(_p(x), N, D, _p(codes), _p(scale))
    return codes, scale


def sparse_attn(q_bf16_bits, kv_bf16_bits, sink, idx, scale: float, lib=None, nthreads=None) -> np.ndarray:
    """float64 [T, H, D] attention output.  q: uint16 bf16 bits [T, H, D]; kv: uint16 bf16 bits
    [N, D]; sink: float32 [H] or None; idx: int32 [T, K] (-1 = no key)."""
    lib = lib or _load()
    q = _c(q_bf16_bits, np.uint16)
    T, H, D = q.shape
    kv = _c(kv_bf16_bits, np.uint16)
    N = kv.shape[0]
    assert kv.shape == (N, D)
    idx = _c(idx, np.int32)
    K = idx.shape[1] if idx.ndim == 2 else 0
    assert idx.shape == (T, K)
    sk = None if sink is None else _c(sink, np.float32)
    assert sk is None or sk.shape == (H,)
    out = np.empty((T, H, D), dtype=np.float64)
    rc = lib.oracle_sparse_attn(_p(q), _p(kv), None if sk is None else _p(sk), _p(idx), T, N, H, D, K,
                                float(scale), _p(out), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle_sparse_attn rejected its arguments (index out of range?)")
    return out


def sparse_attn_bwd(q_bf16_bits, kv_bf16_bits, sink, idx, do_bf16_bits, scale: float, lib=None, nthreads=None):
    """Gradients of sparse_attn for the loss sum(do * o), in float64: (dq [T, H, D], dkv [N, D],
    dsink [H] or None).  do: uint16 bf16 bits [T, H, D]; the other arguments as in sparse_attn."""
    lib = lib or _load()
    q = _c(q_bf16_bits, np.uint16)
    T, H, D = q.shape
    kv = _c(kv_bf16_bits, np.uint16)
    N = kv.shape[0]
    assert kv.shape == (N, D)
    idx = _c(idx, np.int32)
    K = idx.shape[1] if idx.ndim == 2 else 0
    assert idx.shape == (T, K)
    do = _c(do_bf16_bits, np.uint16)
    assert do.shape == (T, H, D)
    sk = None if sink is None else _c(sink, np.float32)
    assert sk is None or sk.shape == (H,)
    dq = np.empty((T, H, D), dtype=np.float64)
    dkv = np.empty((N, D), dtype=np.float64)
    dsink = None if sk is None else np.empty(H, dtype=np.float64)
    rc = lib.oracle_sparse_attn_bwd(_p(q), _p(kv), None if sk is None else _p(sk), _p(idx), _p(do), T, N, H, D, K,
                                    float(scale), _p(dq), _p(dkv), None if dsink is None else _p(dsink),
                                    nthreads or threads())
    if rc != 0:
        raise ValueError("oracle_sparse_attn_bwd rejected its arguments (index out of range?)")
    return dq, dkv, dsink


@dataclass
class RowScores:
    """Oracle scores of selected query rows, stored compactly (window entries only)."""

    rows: np.ndarray  # int64 [R] query rows
    lo: np.ndarray  # int64 [R] first key of each window
    length: np.ndarray  # int64 [R] window length
    offsets: np.ndarray  # int64 [R] start of each row in `flat`
    flat: np.ndarray  # float64 [sum(length)]

    def row(self, r: int) -> np.ndarray:
        """Scores of keys lo[r] .. lo[r]+length[r]-1 of the r-th selected row."""
        o = int(self.offsets[r])
        return self.flat[o:o + int(self.length[r])]

    def dense(self, N: int) -> np.ndarray:
        """[R, N] array with NaN outside each window (small problems only)."""
        out = np.full((len(self.rows), N), np.nan)
        for r in range(len(self.rows)):
            lo = int(self.lo[r])
            out[r, lo:lo + int(self.length[r])] = self.row(r)
        return out


def index_score(q, w, k, k_scale, ks, ke, rows=None, lib=None, nthreads=None) -> RowScores:
    """score[t, j] for t in `rows` (default: all), j in the clamped window of t, in float64.

    Shapes: q uint8 [T, H, D] e4m3 codes, w float32 [T, H], k uint8 [N, D] e4m3 codes,
    k_scale float32 [N], ks / ke int32 [T].
    """
    lib = lib or _load()
    q = _c(q, np.uint8)
    T, H, D = q.shape
    k = _c(k, np.uint8)
    N = k.shape[0]
    assert k.shape == (N, D)
    w = _c(w, np.float32)
    assert w.shape == (T, H)
    k_scale = _c(k_scale, np.float32)
    assert k_scale.shape == (N,)
    ks = _c(ks, np.int32)
    ke = _c(ke, np.int32)
    rows = np.arange(T, dtype=np.int64) if rows is None else _c(rows, np.int64)
    R = len(rows)
    lo = np.empty(R, dtype=np.int64)
    length = np.empty(R, dtype=np.int64)
    if lib.oracle_window_lengths(_p(ks), _p(ke), T, N, _p(rows), R, _p(lo), _p(length)) != 0:
        raise ValueError("bad rows")
    offsets = np.zeros(R, dtype=np.int64)
    if R > 1:
        offsets[1:] = np.cumsum(length)[:-1]
    flat = np.empty(int(length.sum()), dtype=np.float64)
    rc = lib.oracle_index_score(_p(q), _p(w), _p(k), _p(k_scale), _p(ks), _p(ke), T, N, H, D, _p(rows), R,
                                _p(offsets), _p(flat), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle_index_score rejected its arguments")
    return RowScores(rows=rows, lo=lo, length=length, offsets=offsets, flat=flat)


def topk(scores: RowScores, k: int, lib=None, nthreads=None) -> np.ndarray:
    """int32 [R, k]: top-k key indices of each oracle row, ascending, -1 padded."""
    lib = lib or _load()
    R = len(scores.rows)
    idx = np.empty((R, k), dtype=np.int32)
    rc = lib.oracle_topk_compact(_p(scores.flat), _p(scores.offsets), _p(scores.lo), _p(scores.length), R, k,
                                 _p(idx), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle_topk_compact rejected its arguments (NaN score?)")
    return idx


def topk_dense(scores, ks, ke, k: int, lib=None, nthreads=None) -> np.ndarray:
    """Top-k over dense score rows [R, N] (float32 or float64) with per-row windows ks/ke [R].

    Only in-window entries are read, so a GPU logits buffer whose out-of-window entries are
    unspecified can be passed as is.
    """
    lib = lib or _load()
    s = np.asarray(scores)
    if s.dtype == np.float32:
        fn = lib.oracle_topk_f32
    else:
        s = s.astype(np.float64, copy=False)
        fn = lib.oracle_topk_f64
    s = np.ascontiguousarray(s)
    R, N = s.shape
    ks = _c(ks, np.int32)
    ke = _c(ke, np.int32)
    assert ks.shape == (R,) and ke.shape == (R,)
    idx = np.empty((R, k), dtype=np.int32)
    rc = fn(_p(s), N, _p(ks), _p(ke), R, N, k, _p(idx), nthreads or threads())
    if rc != 0:
        raise ValueError("oracle top-k rejected its arguments (NaN score in a window?)")
    return idx


def score_and_topk(wl, rows=None, nthreads=None):
    """(RowScores, idx) of a workloads.Workload for the given rows (default: all)."""
    sc = index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows, nthreads=nthreads)
    return sc, topk(sc, wl.topk, nthreads=nthreads)
