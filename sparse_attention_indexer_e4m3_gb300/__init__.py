"""GB300-native FP8 lightning indexer and exact top-k selector.

Python binding of the C ABI in ``include/dsa.h`` (library ``libdsa_gb300.so``, built in-tree by
``sparse_attention_indexer_e4m3_gb300.build``).  This module only marshals arguments: it checks
torch tensors, passes their device pointers and the current CUDA stream, and raises
``DsaError`` on a non-OK status.  Every step of the computation runs in the library's kernels;
there is no fallback path.  If the library has not been built, every call raises.

    score[t, j] = k_scale[j] * sum_h relu(q[t, h] . k[j]) * w[t, h],   ks[t] <= j < ke[t]
    idx[t]      = the topk keys of largest score in the window, ascending, -1 padded
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "DsaError", "library_path", "load", "index_score", "index_score_kres", "index_score_kres_workspace_size", "topk",
    "index_topk", "index_topk_plan", "index_topk_run", "topk_workspace_size",
    "index_topk_workspace_size", "get_device_error", "status_string", "version", "MAX_TOPK", "SUPPORTED_H",
    "SUPPORTED_D",
]

MAX_TOPK = 2048
SUPPORTED_H = (4, 8, 16, 32, 64)
SUPPORTED_D = (64, 128)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libdsa_gb300.so"
_lib = None
_lock = threading.Lock()

DSA_OK = 0
_STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
           4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT"}


class DsaError(RuntimeError):
    """A non-OK status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load():
    """Load libdsa_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m sparse_attention_indexer_e4m3_gb300.build`")
            lib = ctypes.CDLL(path)
            p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.dsa_index_score.argtypes = [p, p, p, p, p, p, i, i, i, i, p, p]
            lib.dsa_index_score.restype = i
            lib.dsa_index_score_kres_workspace_size.argtypes = [i, i, i, i]
            lib.dsa_index_score_kres_workspace_size.restype = sz
            lib.dsa_index_score_kres.argtypes = [p, p, p, p, p, p, i, i, i, i, p, p, sz, p]
            lib.dsa_index_score_kres.restype = i
            lib.dsa_topk_workspace_size.argtypes = [i, i, i]
            lib.dsa_topk_workspace_size.restype = sz
            lib.dsa_topk.argtypes = [p, p, p, i, i, i, p, p, sz, p]
            lib.dsa_topk.restype = i
            lib.dsa_index_topk_workspace_size.argtypes = [i, i, i, i, i]
            lib.dsa_index_topk_workspace_size.restype = sz
            lib.dsa_index_topk.argtypes = [p, p, p, p, p, p, i, i, i, i, i, p, p, sz, p]
            lib.dsa_index_topk.restype = i
            lib.dsa_index_topk_plan.argtypes = [p, p, i, i, i, i, i, p, sz, p]
            lib.dsa_index_topk_plan.restype = i
            lib.dsa_index_topk_run.argtypes = [p, p, p, p, p, p, i, i, i, i, i, p, p, sz, p]
            lib.dsa_index_topk_run.restype = i
            lib.dsa_get_device_error.argtypes = [p]
            lib.dsa_get_device_error.restype = i
            lib.dsa_quantize_k.argtypes = [p, i, i, p, p, p]
            lib.dsa_quantize_k.restype = i
            lib.dsa_sparse_attn.argtypes = [p, p, p, p, i, i, i, i, i, ctypes.c_float, p, p, p]
            lib.dsa_sparse_attn_bwd.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, ctypes.c_float, p, p, p, p]
            lib.dsa_sparse_attn_bwd.restype = i
            lib.dsa_sparse_attn.restype = i
            lib.dsa_check_bounded_wait.argtypes = [p, p]
            lib.dsa_check_bounded_wait.restype = i
            lib.dsa_status_string.argtypes = [i]
            lib.dsa_status_string.restype = ctypes.c_char_p
            lib.dsa_version.argtypes = []
            lib.dsa_version.restype = i
            _lib = lib
    return _lib


def _torch():
    import torch

    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev(t, name, dtypes):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _shape(t, name, shape):
    """Raise unless tensor t has exactly this shape (caller buffers are never written past)."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


def status_string(status: int) -> str:
    return load().dsa_status_string(status).decode()


def version() -> int:
    return load().dsa_version()


def _inputs(q, w, k, k_scale, ks, ke):
    torch = _torch()
    q = _dev(q, "q", (torch.uint8,))
    k = _dev(k, "k", (torch.uint8,))
    w = _dev(w, "w", (torch.float32,))
    k_scale = _dev(k_scale, "k_scale", (torch.float32,))
    ks = _dev(ks, "ks", (torch.int32,))
    ke = _dev(ke, "ke", (torch.int32,))
    if q.dim() != 3 or k.dim() != 2:
        raise ValueError("q must be [T, H, D] and k must be [N, D]")
    T, H, D = q.shape
    N = k.shape[0]
    if k.shape[1] != D or tuple(w.shape) != (T, H) or tuple(k_scale.shape) != (N,):
        raise ValueError("shape mismatch among q [T,H,D], w [T,H], k [N,D], k_scale [N]")
    if tuple(ks.shape) != (T,) or tuple(ke.shape) != (T,):
        raise ValueError("ks and ke must be [T]")
    return q, w, k, k_scale, ks, ke, T, N, H, D


def index_score(q, w, k, k_scale, ks, ke, logits=None, stream=None):
    """fp32 logits [T, N]; only in-window entries are written (others keep their value)."""
    torch = _torch()
    q, w, k, k_scale, ks, ke, T, N, H, D = _inputs(q, w, k, k_scale, ks, ke)
    if logits is None:
        logits = torch.empty((T, N), dtype=torch.float32, device=q.device)
    logits = _dev(logits, "logits", (torch.float32,))
    if tuple(logits.shape) != (T, N):
        raise ValueError("logits must be [T, N]")
    st = load().dsa_index_score(q.data_ptr(), w.data_ptr(), k.data_ptr(), k_scale.data_ptr(), ks.data_ptr(),
                                ke.data_ptr(), T, N, H, D, logits.data_ptr(), _stream_ptr(stream))
    _check(st, "dsa_index_score")
    return logits


def index_score_kres_workspace_size(T: int, N: int, H: int, D: int) -> int:
    return int(load().dsa_index_score_kres_workspace_size(T, N, H, D))


def index_score_kres(q, w, k, k_scale, ks, ke, logits=None, workspace=None, stream=None):
    """index_score with the key tile resident and the query blocks streamed (same scores, same
    output contract); w must be 16-byte aligned."""
    torch = _torch()
    q, w, k, k_scale, ks, ke, T, N, H, D = _inputs(q, w, k, k_scale, ks, ke)
    if logits is None:
        logits = torch.empty((T, N), dtype=torch.float32, device=q.device)
    logits = _dev(logits, "logits", (torch.float32,))
    if tuple(logits.shape) != (T, N):
        raise ValueError("logits must be [T, N]")
    ws, nbytes = _workspace(index_score_kres_workspace_size(T, N, H, D), workspace, q.device)
    st = load().dsa_index_score_kres(q.data_ptr(), w.data_ptr(), k.data_ptr(), k_scale.data_ptr(), ks.data_ptr(),
                                     ke.data_ptr(), T, N, H, D, logits.data_ptr(),
                                     ws.data_ptr() if ws is not None else None, nbytes, _stream_ptr(stream))
    _check(st, "dsa_index_score_kres")
    return logits


def topk_workspace_size(T: int, N: int, k: int) -> int:
    return int(load().dsa_topk_workspace_size(T, N, k))


def index_topk_workspace_size(T: int, N: int, H: int, D: int, k: int) -> int:
    return int(load().dsa_index_topk_workspace_size(T, N, H, D, k))


def _workspace(nbytes, workspace, device):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    workspace = _dev(workspace, "workspace", (torch.uint8,))
    return workspace, workspace.numel()


def topk(logits, ks, ke, k: int, idx=None, workspace=None, stream=None):
    """int32 [T, k] top-k key indices per row of logits [T, N], ascending, -1 padded."""
    torch = _torch()
    logits = _dev(logits, "logits", (torch.float32,))
    ks = _dev(ks, "ks", (torch.int32,))
    ke = _dev(ke, "ke", (torch.int32,))
    if logits.dim() != 2:
        raise ValueError("logits must be [T, N]")
    T, N = logits.shape
    _shape(ks, "ks", (T,))
    _shape(ke, "ke", (T,))
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    idx = _dev(idx, "idx", (torch.int32,))
    _shape(idx, "idx", (T, k))
    ws, wsb = _workspace(topk_workspace_size(T, N, k), workspace, logits.device)
    st = load().dsa_topk(logits.data_ptr(), ks.data_ptr(), ke.data_ptr(), T, N, k, idx.data_ptr(),
                         None if ws is None else ws.data_ptr(), wsb, _stream_ptr(stream))
    _check(st, "dsa_topk")
    return idx


def index_topk(q, w, k, k_scale, ks, ke, topk_k: int, idx=None, workspace=None, stream=None):
    """Fused scorer + selector: int32 [T, topk_k] without materialising the [T, N] logits."""
    torch = _torch()
    q, w, k, k_scale, ks, ke, T, N, H, D = _inputs(q, w, k, k_scale, ks, ke)
    if idx is None:
        idx = torch.empty((T, topk_k), dtype=torch.int32, device=q.device)
    idx = _dev(idx, "idx", (torch.int32,))
    _shape(idx, "idx", (T, topk_k))
    need = index_topk_workspace_size(T, N, H, D, topk_k)
    ws, wsb = _workspace(need, workspace, q.device)
    st = load().dsa_index_topk(q.data_ptr(), w.data_ptr(), k.data_ptr(), k_scale.data_ptr(), ks.data_ptr(),
                               ke.data_ptr(), T, N, H, D, topk_k, idx.data_ptr(),
                               None if ws is None else ws.data_ptr(), wsb, _stream_ptr(stream))
    _check(st, "dsa_index_topk")
    return idx


def index_topk_plan(ks, ke, N: int, H: int, D: int, topk_k: int, workspace=None, stream=None):
    """Plan the fused path for windows ks / ke; returns the workspace holding the plan."""
    torch = _torch()
    ks = _dev(ks, "ks", (torch.int32,))
    ke = _dev(ke, "ke", (torch.int32,))
    if ks.dim() != 1:
        raise ValueError("ks must be [T]")
    T = ks.shape[0]
    _shape(ke, "ke", (T,))
    need = index_topk_workspace_size(T, N, H, D, topk_k)
    ws, wsb = _workspace(need, workspace, ks.device)
    st = load().dsa_index_topk_plan(ks.data_ptr(), ke.data_ptr(), T, N, H, D, topk_k,
                                    None if ws is None else ws.data_ptr(), wsb, _stream_ptr(stream))
    _check(st, "dsa_index_topk_plan")
    return ws


def index_topk_run(q, w, k, k_scale, ks, ke, topk_k: int, workspace, idx=None, stream=None):
    """Run the fused path with a plan made by index_topk_plan for the same ks / ke / shapes."""
    torch = _torch()
    q, w, k, k_scale, ks, ke, T, N, H, D = _inputs(q, w, k, k_scale, ks, ke)
    if idx is None:
        idx = torch.empty((T, topk_k), dtype=torch.int32, device=q.device)
    idx = _dev(idx, "idx", (torch.int32,))
    _shape(idx, "idx", (T, topk_k))
    ws = None if workspace is None else _dev(workspace, "workspace", (torch.uint8,))
    st = load().dsa_index_topk_run(q.data_ptr(), w.data_ptr(), k.data_ptr(), k_scale.data_ptr(), ks.data_ptr(),
                                   ke.data_ptr(), T, N, H, D, topk_k, idx.data_ptr(),
                                   None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
                                   _stream_ptr(stream))
    _check(st, "dsa_index_topk_run")
    return idx


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().dsa_get_device_error(_stream_ptr(stream)))


def quantize_k(k, codes=None, scale=None, stream=None):
    """e4m3 quantise-on-write of key rows: bf16 [N, D] -> (uint8 codes [N, D], fp32 scales [N])."""
    torch = _torch()
    k = _dev(k, "k", (torch.bfloat16,))
    if k.dim() != 2:
        raise ValueError("k must be [N, D]")
    N, D = k.shape
    if codes is None:
        codes = torch.empty((N, D), dtype=torch.uint8, device=k.device)
    if scale is None:
        scale = torch.empty(N, dtype=torch.float32, device=k.device)
    codes = _dev(codes, "codes", (torch.uint8,))
    scale = _dev(scale, "scale", (torch.float32,))
    _shape(codes, "codes", (N, D))
    _shape(scale, "scale", (N,))
    _check(load().dsa_quantize_k(k.data_ptr(), N, D, codes.data_ptr(), scale.data_ptr(), _stream_ptr(stream)),
           "dsa_quantize_k")
    return codes, scale


def sparse_attn(q, kv, idx, attn_sink=None, scale=None, out=None, lse=None, stream=None):
    """Attention of each query row over its selected keys: q bf16 [T, H, D], kv bf16 [N, D]
    (keys = values), idx int32 [T, K] (-1 = none), attn_sink fp32 [H] or None, scale default
    1 / sqrt(D).  Returns bf16 [T, H, D]; with lse (fp32 [T, H]) given, also writes the natural
    log of each softmax denominator into it (what sparse_attn_bwd takes)."""
    torch = _torch()
    q = _dev(q, "q", (torch.bfloat16,))
    kv = _dev(kv, "kv", (torch.bfloat16,))
    idx = _dev(idx, "idx", (torch.int32,))
    if q.dim() != 3 or kv.dim() != 2 or idx.dim() != 2:
        raise ValueError("shapes: q [T, H, D], kv [N, D], idx [T, K]")
    T, H, D = q.shape
    N = kv.shape[0]
    if kv.shape[1] != D or idx.shape[0] != T:
        raise ValueError("shapes: q [T, H, D], kv [N, D], idx [T, K]")
    sink_ptr = None
    if attn_sink is not None:
        attn_sink = _dev(attn_sink, "attn_sink", (torch.float32,))
        if attn_sink.shape != (H,):
            raise ValueError("attn_sink must be [H]")
        sink_ptr = attn_sink.data_ptr()
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q.device)
    out = _dev(out, "out", (torch.bfloat16,))
    _shape(out, "out", (T, H, D))
    lse_ptr = None
    if lse is not None:
        lse = _dev(lse, "lse", (torch.float32,))
        _shape(lse, "lse", (T, H))
        lse_ptr = lse.data_ptr()
    sc = float(scale) if scale is not None else 1.0 / float(D) ** 0.5
    _check(load().dsa_sparse_attn(q.data_ptr(), kv.data_ptr(), sink_ptr, idx.data_ptr(), T, N, H, D, idx.shape[1],
                                  sc, out.data_ptr(), lse_ptr, _stream_ptr(stream)), "dsa_sparse_attn")
    return out


def sparse_attn_bwd(q, kv, idx, out, lse, dout, attn_sink=None, scale=None, dq=None, dkv=None, dsink=None,
                    stream=None):
    """Gradients of sparse_attn for the loss sum(dout * out): returns (dq fp32 [T, H, D], dkv fp32
    [N, D], dsink fp32 [H] or None).  out and lse are the forward's outputs (bf16 [T, H, D] and
    fp32 [T, H]), dout bf16 [T, H, D]; the other arguments as passed to sparse_attn."""
    torch = _torch()
    q = _dev(q, "q", (torch.bfloat16,))
    kv = _dev(kv, "kv", (torch.bfloat16,))
    idx = _dev(idx, "idx", (torch.int32,))
    if q.dim() != 3 or kv.dim() != 2 or idx.dim() != 2:
        raise ValueError("shapes: q [T, H, D], kv [N, D], idx [T, K]")
    T, H, D = q.shape
    N = kv.shape[0]
    if kv.shape[1] != D or idx.shape[0] != T:
        raise ValueError("shapes: q [T, H, D], kv [N, D], idx [T, K]")
    out = _dev(out, "out", (torch.bfloat16,))
    _shape(out, "out", (T, H, D))
    dout = _dev(dout, "dout", (torch.bfloat16,))
    _shape(dout, "dout", (T, H, D))
    lse = _dev(lse, "lse", (torch.float32,))
    _shape(lse, "lse", (T, H))
    sink_ptr = None
    if attn_sink is not None:
        attn_sink = _dev(attn_sink, "attn_sink", (torch.float32,))
        if attn_sink.shape != (H,):
            raise ValueError("attn_sink must be [H]")
        sink_ptr = attn_sink.data_ptr()
        if dsink is None:
            dsink = torch.empty(H, dtype=torch.float32, device=q.device)
    if dq is None:
        dq = torch.empty((T, H, D), dtype=torch.float32, device=q.device)
    if dkv is None:
        dkv = torch.empty((N, D), dtype=torch.float32, device=q.device)
    dq = _dev(dq, "dq", (torch.float32,))
    _shape(dq, "dq", (T, H, D))
    dkv = _dev(dkv, "dkv", (torch.float32,))
    _shape(dkv, "dkv", (N, D))
    dsink_ptr = None
    if dsink is not None:
        dsink = _dev(dsink, "dsink", (torch.float32,))
        _shape(dsink, "dsink", (H,))
        dsink_ptr = dsink.data_ptr()
    sc = float(scale) if scale is not None else 1.0 / float(D) ** 0.5
    _check(load().dsa_sparse_attn_bwd(q.data_ptr(), kv.data_ptr(), sink_ptr, idx.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), dout.data_ptr(), T, N, H, D, idx.shape[1], sc, dq.data_ptr(),
                                      dkv.data_ptr(), dsink_ptr, _stream_ptr(stream)), "dsa_sparse_attn_bwd")
    return dq, dkv, (dsink if attn_sink is not None else None)


def check_bounded_wait(stream=None):
    """Run the bounded-wait self-check; returns the device time (ns) of its expired wait and of
    the wait that returned on the abort flag.  The timeout it records is left for
    get_device_error()."""
    took = (ctypes.c_uint64 * 2)()
    _check(load().dsa_check_bounded_wait(ctypes.cast(took, ctypes.c_void_p), _stream_ptr(stream)), "dsa_check_bounded_wait")
    return int(took[0]), int(took[1])
