"""Python binding of libcsa.so — DeepSeek-V4 compressed attention (CSA / HCA) on B300.

Argument marshalling only: every function checks tensor devices, dtypes and
contiguity, passes raw device pointers and the current CUDA stream to the C ABI
(include/csa.h), and raises RuntimeError with the library's message on failure.
All computation happens in the library's CUDA kernels; there is no fallback.
PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

CSA_F32, CSA_BF16, CSA_E4M3, CSA_BF16_Q_E4M3, CSA_E2M1 = 0, 1, 2, 3, 4
CSA_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT"}
STATUS_CODES = {v: k for k, v in STATUS_NAMES.items()}

EXPORTS = ("csa_version", "csa_last_error", "csa_workspace_size", "csa_compress", "csa_index_scores", "csa_topk",
           "csa_index_topk", "csa_sparse_attend", "hca_attend", "csa_device_status", "csa_index_topk_static",
           "csa_static_status", "csa_debug_set", "swa_workspace_size", "swa_append", "swa_attend",
           "csa_prefill_workspace_size", "csa_prefill_chunked")
CSA_DEBUG_WAIT_LIMIT, CSA_DEBUG_STARVE_INDEXER = 1, 2
STATIC_SCRATCH_BYTES = 8 << 20


class CsaCacheStruct(ctypes.Structure):
    _fields_ = [
        ("m", ctypes.c_int32), ("d", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("d_idx", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("win_dtype", ctypes.c_int32), ("n_win", ctypes.c_int32),
        ("win_cap", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("max_entries", ctypes.c_int64), ("rope_theta", ctypes.c_double),
        ("kv_nope", ctypes.c_void_p), ("kv_scale", ctypes.c_void_p), ("kv_rope", ctypes.c_void_p),
        ("idx_key", ctypes.c_void_p), ("idx_scale", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("win", ctypes.c_void_p), ("pool_state", ctypes.c_void_p), ("n_tokens", ctypes.c_void_p),
        ("idx_dtype", ctypes.c_int32),
    ]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if libcsa.so has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m long_context_attention_05_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        C = ctypes.POINTER(CsaCacheStruct)
        L.csa_version.restype = I
        L.csa_last_error.restype = ctypes.c_char_p
        L.csa_workspace_size.argtypes = [C, I, I, I, I]
        L.csa_workspace_size.restype = SZ
        L.csa_compress.argtypes = [C, I, I, P, P, P, P, P, P, I, P]
        L.csa_index_scores.argtypes = [C, I, I, P, I, P, I, P, I64, P, SZ, P]
        L.csa_topk.argtypes = [C, I, I, P, I64, I, P, P, P, SZ, P]
        L.csa_index_topk.argtypes = [C, I, I, P, I, P, I, I, P, P, P, SZ, P]
        L.csa_index_topk_static.argtypes = [C, I, I, P, I, P, I, I, P, P, P]
        L.csa_sparse_attend.argtypes = [C, I, I, P, I, I, P, P, I, P, I, P, P, SZ, P]
        L.hca_attend.argtypes = [C, I, I, P, I, I, P, P, I, P, P, SZ, P]
        L.csa_device_status.argtypes = [P, ctypes.POINTER(I), P]
        L.csa_static_status.argtypes = [ctypes.POINTER(I), P]
        L.swa_workspace_size.argtypes = [C, I, I, I]
        L.swa_workspace_size.restype = SZ
        L.swa_append.argtypes = [C, I, I, P, I, P]
        L.swa_attend.argtypes = [C, I, I, P, I, I, P, P, I, P, P, SZ, P]
        L.csa_prefill_workspace_size.argtypes = [C, I, I, I]
        L.csa_prefill_workspace_size.restype = SZ
        L.csa_prefill_chunked.argtypes = [C, I, I, I, P, P, P, P, P, P, I, P, I, P, I, P, I, I, P, I, P, I, P, P, SZ, P]
        L.csa_debug_set.argtypes = [I, ctypes.c_longlong]
        for name in EXPORTS:
            if name not in ("csa_version", "csa_last_error", "csa_workspace_size", "swa_workspace_size",
                            "csa_prefill_workspace_size"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != CSA_OK:
        msg = lib().csa_last_error().decode()
        raise RuntimeError(f"{what} failed ({STATUS_NAMES.get(status, status)}): {msg}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise RuntimeError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise RuntimeError("tensor must be contiguous")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return CSA_F32
    if t.dtype == torch.bfloat16:
        return CSA_BF16
    raise RuntimeError(f"unsupported dtype {t.dtype}")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise RuntimeError(f"{name} must be {dtype}, got {t.dtype}")


class Cache:
    """One layer's compressed cache: device tensors plus the C struct that points
    at them.  Tensor names follow include/csa.h."""

    def __init__(self, *, m, d, d_rope, d_idx, kv_dtype, win_dtype, n_win, win_cap, page_size=0,
                 max_pages=0, max_entries=0, rope_theta=10000.0, tensors: Dict[str, torch.Tensor], idx_dtype=0):
        self.t = tensors
        s = CsaCacheStruct()
        s.m, s.d, s.d_rope, s.d_idx = m, d, d_rope, d_idx
        s.kv_dtype, s.win_dtype, s.n_win, s.win_cap = kv_dtype, win_dtype, n_win, win_cap
        s.page_size, s.max_pages, s.max_entries, s.rope_theta = page_size, max_pages, max_entries, rope_theta
        s.idx_dtype = idx_dtype
        for name in ("kv_nope", "kv_scale", "kv_rope", "idx_key", "idx_scale", "page_table", "win",
                     "pool_state", "n_tokens"):
            setattr(s, name, _ptr(tensors.get(name)))
        self.struct = s
        self.m, self.d, self.d_rope, self.d_idx = m, d, d_rope, d_idx
        self.n_win, self.win_cap, self.page_size = n_win, win_cap, page_size
        self.max_entries, self.max_pages = max_entries, max_pages
        self.kv_dtype, self.win_dtype = kv_dtype, win_dtype

    @property
    def ref(self):
        return ctypes.byref(self.struct)

    @property
    def entry_cap(self) -> int:
        return self.max_pages * self.page_size if self.page_size else self.max_entries

    @classmethod
    def from_host(cls, w, arrs: Dict[str, np.ndarray], device="cuda") -> "Cache":
        """Uploads host arrays (synthetic.seeded_cache / empty_cache layout) for workload w."""
        t = {}
        for k, v in arrs.items():
            v = np.ascontiguousarray(v)
            if v.dtype == np.uint16:
                t[k] = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(device)
            else:
                t[k] = torch.from_numpy(v).to(device)
        return cls(m=w.m, d=w.d, d_rope=w.d_rope, d_idx=w.d_idx,
                   kv_dtype=CSA_E4M3 if w.kv_dtype == "e4m3" else CSA_F32,
                   win_dtype=CSA_F32 if w.tok_dtype == "f32" else CSA_BF16,
                   n_win=w.n_win, win_cap=w.win_cap, page_size=w.page_size, max_pages=w.max_pages,
                   max_entries=w.max_entries if not w.page_size else 0, rope_theta=w.theta, tensors=t,
                   idx_dtype=CSA_E2M1 if getattr(w, "idx_dtype", "") == "e2m1" else 0)


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Host array (fp32, bf16 bits as uint16, uint8, ints) -> device tensor."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def version() -> int:
    return lib().csa_version()


def workspace_size(cache: Cache, batch: int, n_q: int, heads: int, k: int) -> int:
    n = lib().csa_workspace_size(cache.ref, batch, n_q, heads, k)
    if n == 0:
        raise RuntimeError("invalid cache geometry: " + lib().csa_last_error().decode())
    return n


def alloc_workspace(cache: Cache, batch: int, n_q: int, heads: int, k: int, device="cuda") -> torch.Tensor:
    n = workspace_size(cache, batch, n_q, heads, k)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _ws(ws: Optional[torch.Tensor]):
    return (None, 0) if ws is None else (_ptr(ws), ws.numel() * ws.element_size())


def csa_compress(cache: Cache, x, gate, pos_bias, idx_x=None, idx_gate=None, idx_pos_bias=None, stream=None):
    """Append x/gate [B, n_new, d] (+ indexer stream [B, n_new, d_idx]) to the cache."""
    B, n_new = x.shape[0], x.shape[1]
    _need(pos_bias, torch.float32, "pos_bias")
    st = lib().csa_compress(cache.ref, B, n_new, _ptr(x), _ptr(gate), _ptr(idx_x), _ptr(idx_gate), _ptr(pos_bias),
                            _ptr(idx_pos_bias), _dtype_code(x), _stream(stream))
    _check(st, "csa_compress")


def _q_idx_code(q_idx, q_fp8):
    """dtype code of the indexer query; q_fp8 selects the query-side FP8 variant (bf16 input)."""
    if q_fp8:
        _need(q_idx, torch.bfloat16, "q_idx (query-side FP8 variant)")
        return CSA_BF16_Q_E4M3
    return _dtype_code(q_idx)


def csa_index_scores(cache: Cache, q_idx, w, scores, ws=None, stream=None, q_fp8=False):
    """scores [B*n_q, stride] fp32 <- sum_h w_h ReLU(q_h . k_j) for visible entries."""
    B, n_q, H_I = q_idx.shape[0], q_idx.shape[1], q_idx.shape[2]
    _need(w, torch.float32, "w")
    _need(scores, torch.float32, "scores")
    p, n = _ws(ws)
    st = lib().csa_index_scores(cache.ref, B, n_q, _ptr(q_idx), _q_idx_code(q_idx, q_fp8), _ptr(w), H_I, _ptr(scores),
                                scores.shape[-1], p, n, _stream(stream))
    _check(st, "csa_index_scores")


def csa_topk(cache: Cache, scores, batch, n_q, k, out_idx, out_count, ws=None, stream=None):
    _need(scores, torch.float32, "scores")
    _need(out_idx, torch.int32, "out_idx")
    _need(out_count, torch.int32, "out_count")
    p, n = _ws(ws)
    st = lib().csa_topk(cache.ref, batch, n_q, _ptr(scores), scores.shape[-1], k, _ptr(out_idx), _ptr(out_count),
                        p, n, _stream(stream))
    _check(st, "csa_topk")


def csa_index_topk(cache: Cache, q_idx, w, k, out_idx, out_count, ws, stream=None, q_fp8=False):
    B, n_q, H_I = q_idx.shape[0], q_idx.shape[1], q_idx.shape[2]
    _need(w, torch.float32, "w")
    _need(out_idx, torch.int32, "out_idx")
    _need(out_count, torch.int32, "out_count")
    p, n = _ws(ws)
    st = lib().csa_index_topk(cache.ref, B, n_q, _ptr(q_idx), _q_idx_code(q_idx, q_fp8), _ptr(w), H_I, k, _ptr(out_idx),
                              _ptr(out_count), p, n, _stream(stream))
    _check(st, "csa_index_topk")


def csa_index_topk_static(cache: Cache, q_idx, w, k, out_idx, out_count, stream=None):
    """csa_index_topk with the library's own static device scratch instead of a
    caller workspace (for callers that cannot allocate; calls must not overlap)."""
    B, n_q, H_I = q_idx.shape[0], q_idx.shape[1], q_idx.shape[2]
    _need(w, torch.float32, "w")
    _need(out_idx, torch.int32, "out_idx")
    _need(out_count, torch.int32, "out_count")
    st = lib().csa_index_topk_static(cache.ref, B, n_q, _ptr(q_idx), _dtype_code(q_idx), _ptr(w), H_I, k,
                                     _ptr(out_idx), _ptr(out_count), _stream(stream))
    _check(st, "csa_index_topk_static")


def csa_sparse_attend(cache: Cache, q, sink, idx, out, out_lse=None, ws=None, stream=None):
    """q [B, n_q, H, d]; idx int32 [B, n_q, k]; out [B, n_q, H, d] (bf16 or fp32)."""
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    _need(sink, torch.float32, "sink")
    _need(idx, torch.int32, "idx")
    p, n = _ws(ws)
    st = lib().csa_sparse_attend(cache.ref, B, n_q, _ptr(q), _dtype_code(q), H, _ptr(sink), _ptr(idx),
                                 idx.shape[-1], _ptr(out), _dtype_code(out), _ptr(out_lse), p, n, _stream(stream))
    _check(st, "csa_sparse_attend")


def hca_attend(cache: Cache, q, sink, out, out_lse=None, ws=None, stream=None):
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    _need(sink, torch.float32, "sink")
    p, n = _ws(ws)
    st = lib().hca_attend(cache.ref, B, n_q, _ptr(q), _dtype_code(q), H, _ptr(sink), _ptr(out), _dtype_code(out),
                          _ptr(out_lse), p, n, _stream(stream))
    _check(st, "hca_attend")


def swa_append(cache: Cache, x, stream=None):
    """Sliding-window-only layer: raw tokens x [B, n_new, d] into the ring (no pooling)."""
    st = lib().swa_append(cache.ref, x.shape[0], x.shape[1], _ptr(x), _dtype_code(x), _stream(stream))
    _check(st, "swa_append")


def swa_workspace_size(cache: Cache, batch: int, n_q: int, heads: int) -> int:
    n = lib().swa_workspace_size(cache.ref, batch, n_q, heads)
    if n == 0:
        raise RuntimeError("invalid cache geometry: " + lib().csa_last_error().decode())
    return n


def swa_attend(cache: Cache, q, sink, out, out_lse=None, ws=None, stream=None):
    """Attention over the window tokens and the sink only (sliding-window-only layer)."""
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    _need(sink, torch.float32, "sink")
    p, n = _ws(ws)
    st = lib().swa_attend(cache.ref, B, n_q, _ptr(q), _dtype_code(q), H, _ptr(sink), _ptr(out), _dtype_code(out),
                          _ptr(out_lse), p, n, _stream(stream))
    _check(st, "swa_attend")


def prefill_workspace_size(cache: Cache, chunk: int, heads: int, k: int) -> int:
    n = lib().csa_prefill_workspace_size(cache.ref, chunk, heads, k)
    if n == 0:
        raise RuntimeError("invalid prefill geometry: " + lib().csa_last_error().decode())
    return n


def csa_prefill_chunked(cache: Cache, chunk, x, gate, pos_bias, idx_x, idx_gate, idx_pos_bias, q_idx, w, q, sink,
                        k, out, out_lse=None, ws=None, stream=None, q_fp8=False):
    """Prefill of x [B, n_new, d] (and the matching indexer stream, queries and outputs)
    in chunks of `chunk` tokens per sequence."""
    B, n_new = x.shape[0], x.shape[1]
    _need(w, torch.float32, "w")
    _need(sink, torch.float32, "sink")
    if ws is None:
        ws = torch.zeros(prefill_workspace_size(cache, min(chunk, n_new), q.shape[2], k), dtype=torch.uint8,
                         device=x.device)
    p, n = _ws(ws)
    st = lib().csa_prefill_chunked(cache.ref, B, n_new, chunk, _ptr(x), _ptr(gate), _ptr(idx_x), _ptr(idx_gate),
                                   _ptr(pos_bias), _ptr(idx_pos_bias), _dtype_code(x), _ptr(q_idx),
                                   _q_idx_code(q_idx, q_fp8), _ptr(w), q_idx.shape[2], _ptr(q), _dtype_code(q),
                                   q.shape[2], _ptr(sink), k, _ptr(out), _dtype_code(out), _ptr(out_lse), p, n,
                                   _stream(stream))
    _check(st, "csa_prefill_chunked")


def device_status(ws: torch.Tensor, stream=None) -> int:
    """Reads and clears the workspace's device status word (0 = fine, 5 = a bounded wait gave up)."""
    v = ctypes.c_int(0)
    _check(lib().csa_device_status(_ptr(ws), ctypes.byref(v), _stream(stream)), "csa_device_status")
    return v.value


def static_status(stream=None) -> int:
    """Reads and clears the status word of csa_index_topk_static's scratch (current device)."""
    v = ctypes.c_int(0)
    _check(lib().csa_static_status(ctypes.byref(v), _stream(stream)), "csa_static_status")
    return v.value


def debug_set(knob: int, value: int) -> None:
    """Failure injection for tests of the indexer's bounded waits (see include/csa.h)."""
    _check(lib().csa_debug_set(knob, int(value)), "csa_debug_set")
