"""The C ABI on the CPU: the library loads, exports every declared entry
point, and rejects bad arguments with a status before touching the GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from rag_precomputed_kv_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvr.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    from rag_precomputed_kv_gb300 import kvr
    return kvr.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"KVR_API\s+[\w\s\*]+?\b(kvr_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kvr_pool_register", "kvr_pool_unregister", "kvr_assemble", "kvr_query_attention",
              "kvr_prefill", "kvr_check", "kvr_status_string", "kvr_last_error", "kvr_attention_path",
              "kvr_set_timing_events"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from rag_precomputed_kv_gb300 import kvr
    for code, name in kvr.STATUS.items():
        assert lib.kvr_status_string(code).decode() == name


def _desc(**kw):
    from rag_precomputed_kv_gb300 import kvr
    d = dict(n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, dtype=kvr.KVR_DTYPE_BF16,
             flags=0, n_entries=4, entry_len=512, k=0x10000, v=0x20000,
             stride=(2 * 2 * 512 * 128, 2 * 512 * 128, 512 * 128, 128), rope_theta=1e6)
    d.update(kw)
    s = d.pop("stride")
    desc = kvr.PoolDesc(**{k: v for k, v in d.items()})
    desc.stride = (ctypes.c_int64 * 4)(*s)
    return desc


def _register(lib, desc):
    h = ctypes.c_void_p()
    st = lib.kvr_pool_register(ctypes.byref(desc), ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("bad,status", [
    (dict(dtype=7), 3), (dict(head_dim=96), 3), (dict(n_q_heads=7), 1), (dict(n_layers=0), 1),
    (dict(n_entries=0), 1), (dict(flags=4), 1), (dict(flags=-1), 1), (dict(k=0), 1), (dict(k=0x10008), 1),
    (dict(rope_theta=0.5), 1), (dict(stride=(8, 8, 8, 12)), 1), (dict(stride=(-8, 8, 8, 8)), 1),
])
def test_register_rejects_bad_descriptors(lib, bad, status):
    st, h = _register(lib, _desc(**bad))
    assert st == status and not h.value
    assert lib.kvr_last_error().decode()


def test_reserve_rejects_bad_limits_before_any_cuda_call(lib):
    st, h = _register(lib, _desc())
    assert st == 0 and h.value
    try:
        assert lib.kvr_pool_reserve(None, 1, 1, 0, 1) == 1
        for bad in ((-1, 0, 0, 0), (0, -1, 0, 0), (0, 0, -1, 0), (0, 0, 0, -1), (0, 0, 0, 1 << 31)):
            assert lib.kvr_pool_reserve(h, *bad) == 1, bad
            assert "reservation" in lib.kvr_last_error().decode()
    finally:
        lib.kvr_pool_unregister(h)


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.kvr_pool_register(None, ctypes.byref(h)) == 1
    assert lib.kvr_assemble(None, 1, None, None, None, 0, None, None, None, None, None, None, 0, None) == 1
    assert lib.kvr_query_attention(None, 1, None, None, None, None, None, None, None, None, None,
                                   ctypes.c_float(0), None) == 1
    assert lib.kvr_prefill(None, 1, None, None, None, 0, None, None, None, None, None, None, 0,
                           None, None, None, None, None, ctypes.c_float(0), None) == 1
    assert lib.kvr_selftest_wait(None, 1000, None) == 1
    assert lib.kvr_pool_unregister(None) == 0


def _assemble(lib, h, spans, span_offsets, cache_offsets, locals_=None, n_locals=0, flags=0,
              cache=0x100000):
    from rag_precomputed_kv_gb300 import kvr
    so = np.ascontiguousarray(span_offsets, np.int32)
    sp = np.ascontiguousarray(spans, np.int32).reshape(-1, 3)
    co = np.ascontiguousarray(cache_offsets, np.int64)
    plen = np.zeros(len(so), np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = lib.kvr_assemble(h, len(so) - 1, p(so), p(sp) if sp.size else None, locals_, n_locals,
                          p(co), cache, cache, None, None, p(plen), flags, None)
    return st, plen


def test_empty_and_negative_batches(lib):
    """A batch of no requests is a no-op (no table is read, no GPU work); a
    negative batch is an invalid argument -- for each of the three calls."""
    st, h = _register(lib, _desc())
    assert st == 0
    try:
        f0 = ctypes.c_float(0)
        for batch, want in ((0, 0), (-1, 1)):
            assert lib.kvr_assemble(h, batch, None, None, None, 0, None, None, None, None, None, None, 0,
                                    None) == want
            assert lib.kvr_query_attention(h, batch, None, None, None, None, None, None, None, None, None,
                                           f0, None) == want
            assert lib.kvr_prefill(h, batch, None, None, None, 0, None, None, None, None, None, None, 0,
                                   None, None, None, None, None, f0, None) == want
    finally:
        lib.kvr_pool_unregister(h)


def test_assemble_validates_spans_before_any_gpu_work(lib):
    st, h = _register(lib, _desc())
    assert st == 0
    try:
        # unknown pool entry, span past the entry end, inverted span, local without locals
        for spans in ([[4, 0, 8]], [[0, 500, 513]], [[0, 9, 8]], [[-1, 0, 1]], [[(1 << 30) | 0, 0, 4]]):
            st, _ = _assemble(lib, h, spans, [0, 1], [0, 1000])
            assert st == 2, spans
        # prefix longer than the cache block
        st, _ = _assemble(lib, h, [[0, 0, 512], [1, 0, 512]], [0, 2], [0, 1000])
        assert st == 2
        # non-monotone offsets, bad flags
        assert _assemble(lib, h, [[0, 0, 8]], [1, 1], [0, 100])[0] == 1
        assert _assemble(lib, h, [[0, 0, 8]], [0, 1], [10, 5])[0] == 1
        assert _assemble(lib, h, [[0, 0, 8]], [0, 1], [0, 100], flags=4)[0] == 1
        # misaligned cache pointer
        assert _assemble(lib, h, [[0, 0, 8]], [0, 1], [0, 100], cache=0x100004)[0] == 1
        # only empty spans: nothing to launch, prefix lengths are still reported
        st, plen = _assemble(lib, h, [[0, 3, 3], [2, 0, 0]], [0, 1, 2], [0, 10, 20])
        assert st == 0 and plen[:2].tolist() == [0, 0]
    finally:
        lib.kvr_pool_unregister(h)


def test_query_attention_validates_capacity(lib):
    st, h = _register(lib, _desc())
    assert st == 0
    try:
        co = np.array([0, 100], np.int64)
        pl = np.array([90], np.int32)
        qo = np.array([0, 16], np.int32)
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        buf = 0x100000
        st = lib.kvr_query_attention(h, 1, p(co), p(pl), p(qo), buf, buf, buf, buf, buf, buf,
                                     ctypes.c_float(0), None)
        assert st == 2                         # 90 + 16 > 100 rows
        st = lib.kvr_query_attention(h, 1, p(co), p(pl), p(qo), buf + 2, buf, buf, buf, buf, buf,
                                     ctypes.c_float(0), None)
        assert st == 1                         # misaligned q
        st = lib.kvr_query_attention(h, 1, p(co), p(pl), p(qo), buf, buf, buf, buf, buf, buf,
                                     ctypes.c_float(-1.0), None)
        assert st == 1                         # negative scale
    finally:
        lib.kvr_pool_unregister(h)


def test_no_gpu_means_cuda_error_not_a_crash(lib):
    """With valid arguments and no GPU, the first call that needs the device
    reports KVR_ERR_CUDA (no CPU fallback exists)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _register(lib, _desc())
    try:
        st, _ = _assemble(lib, h, [[0, 0, 8]], [0, 1], [0, 100])
        assert st == 4
    finally:
        lib.kvr_pool_unregister(h)


def _prefill(lib, h, spans, span_offsets, cache_offsets, q_offsets, q=0x200000, cache=0x100000,
             flags=0, scale=0.0):
    so = np.ascontiguousarray(span_offsets, np.int32)
    sp = np.ascontiguousarray(spans, np.int32).reshape(-1, 3)
    co = np.ascontiguousarray(cache_offsets, np.int64)
    qo = np.ascontiguousarray(q_offsets, np.int32)
    plen = np.full(len(so), -7, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = lib.kvr_prefill(h, len(so) - 1, p(so), p(sp) if sp.size else None, None, 0, p(co),
                         cache, cache, None, None, p(plen), flags, p(qo), q, q, q, q,
                         ctypes.c_float(scale), None)
    return st, plen


def test_prefill_checks_both_halves_before_any_gpu_work(lib):
    """kvr_prefill rejects a bad stitch and a bad query half alike, without a
    GPU and before writing its prefix-length output."""
    st, h = _register(lib, _desc())
    assert st == 0
    try:
        # stitch half: unknown entry, span past the end of its entry
        for spans in ([[4, 0, 8]], [[0, 500, 513]]):
            st, plen = _prefill(lib, h, spans, [0, 1], [0, 1000], [0, 4])
            assert st == 2 and plen[0] == -7, spans
        # query half: the stitched prefix (512) + 16 query rows overflow 520 rows
        st, plen = _prefill(lib, h, [[0, 0, 512]], [0, 1], [0, 520], [0, 16])
        assert st == 2 and plen[0] == -7
        # query half: misaligned q, negative scale, decreasing q_offsets
        assert _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4], q=0x200002)[0] == 1
        assert _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4], scale=-1.0)[0] == 1
        assert _prefill(lib, h, [[0, 0, 8], [1, 0, 8]], [0, 1, 2], [0, 100, 200], [0, 4, 2])[0] == 1
        # nothing to do at all: empty spans and no query tokens; P_b reported
        st, plen = _prefill(lib, h, [[0, 3, 3]], [0, 1], [0, 10], [0, 0])
        assert st == 0 and plen[0] == 0
    finally:
        lib.kvr_pool_unregister(h)


def test_prefill_without_gpu_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _register(lib, _desc())
    try:
        st, plen = _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4])
        assert st == 4 and plen[0] == 8
    finally:
        lib.kvr_pool_unregister(h)


def test_prefill_skip_prefix_cache_checks_the_pool_layout(lib):
    """KVR_PREFILL_SKIP_PREFIX_CACHE needs a bf16 pool with head_dim 128: an
    fp32 pool is refused up front; a pool with padded strides passes the
    checks (and, with no GPU here, fails only at the device)."""
    import torch
    from rag_precomputed_kv_gb300 import kvr
    flag = kvr.KVR_PREFILL_SKIP_PREFIX_CACHE
    st, h = _register(lib, _desc(dtype=kvr.KVR_DTYPE_FP32, stride=(2 * 2 * 512 * 128, 2 * 512 * 128, 512 * 128, 128)))
    assert st == 0
    try:
        assert _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4], flags=flag)[0] == 3
    finally:
        lib.kvr_pool_unregister(h)
    if not torch.cuda.is_available():
        st, h = _register(lib, _desc(stride=(2 * 2 * 512 * 128 + 128, 2 * 512 * 128, 512 * 128, 128)))
        assert st == 0
        try:
            assert _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4], flags=flag)[0] == 4
        finally:
            lib.kvr_pool_unregister(h)
    # unknown flag bits are still invalid
    st, h = _register(lib, _desc())
    try:
        assert _prefill(lib, h, [[0, 0, 8]], [0, 1], [0, 100], [0, 4], flags=8)[0] == 1
    finally:
        lib.kvr_pool_unregister(h)
