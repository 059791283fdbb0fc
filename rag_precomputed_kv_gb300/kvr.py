"""Thin ctypes binding of libkvr (include/kvr.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; this module
converts torch tensors to device pointers, host lists to C arrays, and
statuses to exceptions.  There is no fallback: if libkvr.so is missing the
import fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvr.so")

KVR_OK = 0
KVR_DTYPE_BF16 = 0
KVR_DTYPE_FP32 = 1
KVR_SRC_LOCAL = 1 << 30
KVR_POSITIONS_COMPOSITE = 1
KVR_PREFILL_SKIP_PREFIX_CACHE = 2
KVR_POOL_KEYS_UNROTATED = 1
KVR_POOL_ROPE_INTERLEAVED = 2

STATUS = {0: "KVR_OK", 1: "KVR_ERR_INVALID_ARG", 2: "KVR_ERR_OUT_OF_RANGE", 3: "KVR_ERR_UNSUPPORTED",
          4: "KVR_ERR_CUDA", 5: "KVR_ERR_TIMEOUT", 6: "KVR_ERR_DEVICE_CHECK"}

EXPORTED = ("kvr_pool_register", "kvr_pool_unregister", "kvr_assemble", "kvr_query_attention",
            "kvr_prefill", "kvr_check", "kvr_status_string", "kvr_last_error", "kvr_attention_path",
            "kvr_set_timing_events", "kvr_selftest_wait", "kvr_assemble_noalloc", "kvr_pool_reserve")
PATH_UNBOUND, PATH_CUDA_CORES, PATH_TCGEN05 = -1, 0, 1


class KvrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("n_entries", ctypes.c_int64), ("entry_len", ctypes.c_int64),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("stride", ctypes.c_int64 * 4), ("rope_theta", ctypes.c_double)]


class Span(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int32), ("start", ctypes.c_int32), ("end", ctypes.c_int32)]


class LocalSrc(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_int64),
                ("stride", ctypes.c_int64 * 3)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libkvr.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with rag_precomputed_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.kvr_pool_register.argtypes = [ctypes.POINTER(PoolDesc), ctypes.POINTER(vp)]
    lib.kvr_pool_unregister.argtypes = [vp]
    lib.kvr_assemble.argtypes = [vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, ctypes.c_uint32, vp]
    lib.kvr_query_attention.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp]
    lib.kvr_prefill.argtypes = [vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, ctypes.c_uint32,
                                vp, vp, vp, vp, vp, ctypes.c_float, vp]
    lib.kvr_check.argtypes = [vp, vp]
    lib.kvr_assemble_noalloc.argtypes = [ctypes.POINTER(PoolDesc), i32, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                         vp, ctypes.c_uint32, vp]
    lib.kvr_selftest_wait.argtypes = [vp, ctypes.c_uint64, vp]
    lib.kvr_pool_reserve.argtypes = [vp, i32, i32, i32, i64]
    lib.kvr_status_string.restype = ctypes.c_char_p
    lib.kvr_status_string.argtypes = [ctypes.c_int]
    lib.kvr_last_error.restype = ctypes.c_char_p
    lib.kvr_set_timing_events.argtypes = [vp, vp]
    lib.kvr_set_timing_events.restype = ctypes.c_int
    lib.kvr_attention_path.argtypes = [vp]
    lib.kvr_attention_path.restype = ctypes.c_int32
    for name in ("kvr_pool_register", "kvr_pool_unregister", "kvr_assemble", "kvr_query_attention",
                 "kvr_prefill", "kvr_check", "kvr_selftest_wait", "kvr_assemble_noalloc", "kvr_pool_reserve"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _raise(st: int):
    if st != KVR_OK:
        raise KvrError(st, load().kvr_last_error().decode())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _np_ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _span_args(span_offsets, spans, cache_offsets, locals_):
    so = _i32(span_offsets)
    sp = _i32(spans).reshape(-1, 3)
    co = _i64(cache_offsets)
    loc = (LocalSrc * max(1, len(locals_)))()
    for i, (lk, lv) in enumerate(locals_):
        assert lk.stride() == lv.stride() and lk.stride(-1) == 1
        loc[i] = LocalSrc(_ptr(lk), _ptr(lv), lk.shape[2], (ctypes.c_int64 * 3)(*lk.stride()[:3]))
    return so, sp, co, loc, len(so) - 1


def _pool_desc(k, v, n_q_heads: int, rope_theta: float, keys_unrotated: bool, rope_interleaved: bool):
    import torch
    assert k.shape == v.shape and k.stride() == v.stride() and k.dtype == v.dtype
    assert k.stride(-1) == 1
    dt = {torch.bfloat16: KVR_DTYPE_BF16, torch.float32: KVR_DTYPE_FP32}[k.dtype]
    E, L, H, T, D = k.shape
    flags = ((KVR_POOL_KEYS_UNROTATED if keys_unrotated else 0)
             | (KVR_POOL_ROPE_INTERLEAVED if rope_interleaved else 0))
    return PoolDesc(L, n_q_heads, H, D, dt, flags, E, T, _ptr(k), _ptr(v),
                    (ctypes.c_int64 * 4)(*k.stride()[:4]), float(rope_theta))


def assemble_noalloc(k, v, n_q_heads: int, rope_theta: float, span_offsets: Sequence[int], spans,
                     cache_offsets, cache_k, cache_v, locals_=(), pos_ids=None, src_map=None,
                     composite: bool = False, keys_unrotated: bool = False,
                     rope_interleaved: bool = False, stream=None) -> np.ndarray:
    """kvr_assemble_noalloc: kvr_assemble for callers that cannot allocate.

    No pool handle: the pool tensors ``k``, ``v`` are described as for
    :class:`Pool` on every call.  Returns the per-request prefix lengths
    (numpy int32).  The library's fixed scratch is shared by all such calls
    (see the header for its limits and its one-call-at-a-time rule).
    """
    d = _pool_desc(k, v, n_q_heads, rope_theta, keys_unrotated, rope_interleaved)
    so, sp, co, loc, batch = _span_args(span_offsets, spans, cache_offsets, locals_)
    plen = np.zeros(max(batch, 1), np.int32)
    _raise(load().kvr_assemble_noalloc(ctypes.byref(d), batch, _np_ptr(so), _np_ptr(sp) if sp.size else None,
                                       ctypes.cast(loc, ctypes.c_void_p) if len(locals_) else None,
                                       len(locals_), _np_ptr(co), _ptr(cache_k), _ptr(cache_v),
                                       _ptr(pos_ids), _ptr(src_map), _np_ptr(plen),
                                       KVR_POSITIONS_COMPOSITE if composite else 0, _stream_ptr(stream)))
    return plen[:batch]


class Pool:
    """A registered pool of precomputed chunk caches.

    ``k``, ``v``: tensors ``[entries, layers, kv_heads, entry_len, head_dim]`` in
    device memory or pinned host memory (any strides with head_dim contiguous),
    keys rotated at entry-local positions (or, with ``keys_unrotated``, before
    RoPE).  ``rope_interleaved``:
    RoPE pairs are (x_2i, x_2i+1) instead of (x_i, x_i+D/2), for the stored
    keys and every rotation the library makes.  The tensors must outlive the
    pool.
    """

    def __init__(self, k, v, n_q_heads: int, rope_theta: float, keys_unrotated: bool = False,
                 rope_interleaved: bool = False):
        lib = load()
        d = _pool_desc(k, v, n_q_heads, rope_theta, keys_unrotated, rope_interleaved)
        _, L, H, _, D = k.shape
        h = ctypes.c_void_p()
        _raise(lib.kvr_pool_register(ctypes.byref(d), ctypes.byref(h)))
        self._h = h
        self._keep = (k, v)
        self.n_layers, self.n_kv_heads, self.n_q_heads, self.head_dim = L, H, n_q_heads, D
        self.dtype = k.dtype

    def reserve(self, max_batch: int = 0, max_spans: int = 0, max_locals: int = 0, max_query_tokens: int = 0):
        """kvr_pool_reserve: bind the pool to the current device and allocate
        now every staging and scratch buffer that calls within these limits
        need; later calls within them never allocate."""
        _raise(load().kvr_pool_reserve(self._h, int(max_batch), int(max_spans), int(max_locals),
                                       int(max_query_tokens)))

    def close(self):
        if getattr(self, "_h", None):
            load().kvr_pool_unregister(self._h)
            self._h = None

    __del__ = close

    def assemble(self, span_offsets: Sequence[int], spans, cache_offsets, cache_k, cache_v,
                 locals_=(), pos_ids=None, src_map=None, composite: bool = False, stream=None):
        """kvr_assemble; returns the per-request prefix lengths (numpy int32)."""
        so, sp, co, loc, batch = _span_args(span_offsets, spans, cache_offsets, locals_)
        plen = np.zeros(max(batch, 1), np.int32)
        _raise(load().kvr_assemble(self._h, batch, _np_ptr(so), _np_ptr(sp) if sp.size else None,
                                   ctypes.cast(loc, ctypes.c_void_p) if len(locals_) else None,
                                   len(locals_), _np_ptr(co),
                                   _ptr(cache_k), _ptr(cache_v), _ptr(pos_ids), _ptr(src_map),
                                   _np_ptr(plen), KVR_POSITIONS_COMPOSITE if composite else 0,
                                   _stream_ptr(stream)))
        return plen[:batch]

    def prefill(self, span_offsets: Sequence[int], spans, cache_offsets, cache_k, cache_v,
                q_offsets, q, kq, vq, out, locals_=(), pos_ids=None, src_map=None,
                composite: bool = False, softmax_scale: float = 0.0, skip_prefix_cache: bool = False,
                stream=None):
        """kvr_prefill (assemble + query attention in one call); returns the
        per-request prefix lengths (numpy int32).  skip_prefix_cache: the
        attention gathers the prefix from the pool and the cache's prefix rows
        are not written (KVR_PREFILL_SKIP_PREFIX_CACHE)."""
        so, sp, co, loc, batch = _span_args(span_offsets, spans, cache_offsets, locals_)
        qo = _i32(q_offsets)
        plen = np.zeros(max(batch, 1), np.int32)
        _raise(load().kvr_prefill(self._h, batch, _np_ptr(so), _np_ptr(sp) if sp.size else None,
                                  ctypes.cast(loc, ctypes.c_void_p) if len(locals_) else None,
                                  len(locals_), _np_ptr(co),
                                  _ptr(cache_k), _ptr(cache_v), _ptr(pos_ids), _ptr(src_map),
                                  _np_ptr(plen), (KVR_POSITIONS_COMPOSITE if composite else 0) |
                                  (KVR_PREFILL_SKIP_PREFIX_CACHE if skip_prefix_cache else 0),
                                  _np_ptr(qo), _ptr(q), _ptr(kq), _ptr(vq), _ptr(out),
                                  float(softmax_scale), _stream_ptr(stream)))
        return plen[:batch]

    def query_attention(self, cache_offsets, prefix_len, q_offsets, q, kq, vq, cache_k, cache_v,
                        out, softmax_scale: float = 0.0, stream=None):
        """kvr_query_attention (appends the query K/V to the cache, writes out).
        ``q``, ``kq``, ``vq`` and ``out`` may be device or pinned host tensors;
        with one token per request the call is a decode step (one kernel)."""
        co, pl, qo = _i64(cache_offsets), _i32(prefix_len), _i32(q_offsets)
        _raise(load().kvr_query_attention(self._h, len(qo) - 1, _np_ptr(co), _np_ptr(pl), _np_ptr(qo),
                                          _ptr(q), _ptr(kq), _ptr(vq), _ptr(cache_k), _ptr(cache_v),
                                          _ptr(out), float(softmax_scale), _stream_ptr(stream)))

    @property
    def attention_path(self) -> int:
        """PATH_TCGEN05, PATH_CUDA_CORES, or PATH_UNBOUND before the first call."""
        return int(load().kvr_attention_path(self._h))

    def set_timing_events(self, events):
        """Six torch.cuda.Event(enable_timing=True) recorded around the
        assemble, query-append and attention kernels (None turns it off)."""
        if events is None:
            _raise(load().kvr_set_timing_events(self._h, None))
            return
        arr = (ctypes.c_void_p * 6)(*[int(e.cuda_event) for e in events])
        _raise(load().kvr_set_timing_events(self._h, ctypes.cast(arr, ctypes.c_void_p)))

    def selftest_wait(self, limit_ns: int, stream=None):
        """Enqueue a kernel whose bounded wait runs out after ``limit_ns``
        (the library's timeout path); the next :meth:`check` raises
        KVR_ERR_TIMEOUT."""
        _raise(load().kvr_selftest_wait(self._h, int(limit_ns), _stream_ptr(stream)))

    def check(self, stream=None):
        """kvr_check: synchronize and raise on a device-recorded error."""
        _raise(load().kvr_check(self._h, _stream_ptr(stream)))
