"""fp64 CPU oracle for the precomputed-KV RAG hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The
product library (``rag_precomputed_kv_gb300``) never imports, links or runs it,
and this package shares no code with the CUDA path.

What each function follows (page titles and sections):

* :func:`positions` -- CoinRAG blog, section 2.3: the stitched prefix
  ``C_ctx = C_p (+) Rot(C_b1[s1:e1]; D1) (+) ...`` with the new position of
  span i given by the prompt length plus the lengths of the spans before it;
  TurboRAG blog, "Position ID": reordered vs composite positions (Figure 5).
* :func:`rope` -- RoPE rotation R(shift) on half-split pairs (or, with
  ``interleaved``, on adjacent pairs).  CoinRAG blog section 2.3 (``Rot``),
  TurboRAG blog ("RoPE only cares about relative position"; "re-apply RoPE at
  the new position").
* :func:`assemble` -- gather + re-rotate + stitch of one request (CoinRAG
  blog section 2.3; SemPIC page, hit path: re-rotate RoPE keys at the final
  logical positions and interleave request-side inline tokens).
* :func:`query_attention` -- query prefill over the stitched prefix
  (CoinRAG blog section 2.3, ``KV_CoinRAG = C_ctx (+) KV_M(q; C_ctx)``;
  TurboRAG blog, "Attention Mask": the query sees every chunk and itself).

The arithmetic lives in ``kvr_oracle.c`` (plain loops, double precision);
this module only converts arrays and slices sources (library primitives).
Pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvr_oracle.c")
_LIB = os.path.join(_HERE, "libkvr_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _LIB, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    return _LIB


class _Span(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int32), ("start", ctypes.c_int32), ("end", ctypes.c_int32)]


def _bind(lib):
    p = ctypes.c_void_p
    lib.kvo_num_threads.restype = ctypes.c_int
    lib.kvo_positions.restype = ctypes.c_int64
    lib.kvo_positions.argtypes = [ctypes.c_int, p, ctypes.c_int64, ctypes.c_int,
                                  p, p, p, p, p]
    lib.kvo_rope_rows.restype = None
    lib.kvo_rope_rows.argtypes = [ctypes.c_int64, ctypes.c_int, p, p, ctypes.c_double, p]
    lib.kvo_rope_rows_interleaved.restype = None
    lib.kvo_rope_rows_interleaved.argtypes = lib.kvo_rope_rows.argtypes
    lib.kvo_query_attention_units.restype = ctypes.c_int
    lib.kvo_query_attention_units.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              ctypes.c_int, ctypes.c_double, p, p, p, p, p, p]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the oracle from another build of ``kvr_oracle.c`` for the duration
    of the block (the tests build copies with planted mistakes to show that
    the pins catch them)."""
    global _lib
    saved = _lib
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def num_threads() -> int:
    """Threads the oracle's parallel loop uses (OMP_NUM_THREADS or all cores)."""
    return int(_load().kvo_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Positions:
    target: np.ndarray   # int64 [k]  position the first token of span i lands at
    delta: np.ndarray    # int64 [k]  rotation applied to span i (target - start)
    pos: np.ndarray      # int32 [P]  position id of each stitched token
    src_id: np.ndarray   # int32 [P]  source id of each stitched token
    src_tok: np.ndarray  # int32 [P]  token index inside its source
    total: int           # P


def positions(spans, first_pos: int = 0, composite: bool = False) -> Positions:
    """Target positions and per-token maps of one request's span list.

    ``spans``: int array [k, 3] of (src, start, end), half-open.  Reordered
    positions put span i at ``first_pos + sum_{j<i} len_j``; composite
    positions keep the chunk-local ids.
    """
    sp = np.ascontiguousarray(np.asarray(spans, dtype=np.int32).reshape(-1, 3))
    k = sp.shape[0]
    arr = (_Span * max(k, 1))()
    for i in range(k):
        arr[i] = _Span(int(sp[i, 0]), int(sp[i, 1]), int(sp[i, 2]))
    lens = np.maximum(sp[:, 2].astype(np.int64) - sp[:, 1], 0)
    P = int(lens.sum())
    target = np.zeros(max(k, 1), np.int64)
    delta = np.zeros(max(k, 1), np.int64)
    pos = np.zeros(max(P, 1), np.int32)
    sid = np.zeros(max(P, 1), np.int32)
    stok = np.zeros(max(P, 1), np.int32)
    got = _load().kvo_positions(k, ctypes.cast(arr, ctypes.c_void_p), int(first_pos),
                                int(bool(composite)), _ptr(target), _ptr(delta),
                                _ptr(pos), _ptr(sid), _ptr(stok))
    if got < 0:
        raise ValueError("invalid span (start < 0 or end < start)")
    return Positions(target[:k], delta[:k], pos[:got], sid[:got], stok[:got], int(got))


def rope(x, shift, theta: float, interleaved: bool = False) -> np.ndarray:
    """Rotate rows ``x[..., D]`` by ``shift`` (scalar, or one value per row).

    Pairs are (x_i, x_{i+D/2}), or (x_{2i}, x_{2i+1}) with ``interleaved``.
    """
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    sh = np.ascontiguousarray(np.broadcast_to(np.asarray(shift, dtype=np.float64),
                                              x.shape[:-1]).reshape(-1))
    out = np.empty_like(rows)
    lib = _load()
    fn = lib.kvo_rope_rows_interleaved if interleaved else lib.kvo_rope_rows
    fn(rows.shape[0], D, _ptr(rows), _ptr(sh), float(theta), _ptr(out))
    return out.reshape(x.shape)


def assemble(sources, spans, theta: float, first_pos: int = 0, composite: bool = False,
             unrotated=(), interleaved: bool = False):
    """Stitch one request's prefix.

    ``sources`` maps a source id to a pair ``(k, v)`` of arrays
    ``[L, H_kv, n_tokens, D]`` whose keys are rotated at their source-local
    positions 0..n_tokens-1 (any float dtype; converted exactly to fp64).
    Returns ``(K, V, Positions)`` with K, V fp64 ``[L, H_kv, P, D]``: span i's
    keys rotated by ``delta_i``, its values copied.

    Sources named in ``unrotated`` hold their keys before RoPE (TurboRAG
    blog, "Position ID": keep the un-rotated K and apply RoPE at the new
    position when stitching): their tokens are rotated at their positions.
    ``interleaved`` selects the adjacent-pair RoPE layout.
    """
    pz = positions(spans, first_pos, composite)
    sp = np.asarray(spans, dtype=np.int64).reshape(-1, 3)
    first = next(iter(sources.values()))[0]
    L, H, _, D = first.shape
    K = np.zeros((L, H, pz.total, D), np.float64)
    V = np.zeros((L, H, pz.total, D), np.float64)
    row = 0
    for i, (src, s, e) in enumerate(sp):
        n = int(e - s)
        if n <= 0:
            continue
        k_src, v_src = sources[int(src)]
        k_rows = np.asarray(k_src[:, :, s:e, :], dtype=np.float64)
        if int(src) in unrotated:
            at = pz.pos[row:row + n].astype(np.float64)
            K[:, :, row:row + n, :] = rope(k_rows, np.broadcast_to(at, k_rows.shape[:-1]), theta,
                                           interleaved)
        else:
            K[:, :, row:row + n, :] = rope(k_rows, float(pz.delta[i]), theta, interleaved)
        V[:, :, row:row + n, :] = np.asarray(v_src[:, :, s:e, :], dtype=np.float64)
        row += n
    return K, V, pz


def query_attention(kc, vc, q, kq, vq, theta: float, scale: float = 0.0,
                    interleaved: bool = False) -> np.ndarray:
    """Query prefill over stitched prefixes of ``U`` independent units.

    kc, vc: [U, P, D]; q: [U, Lq, G, D]; kq, vq: [U, Lq, D] (query-side
    arrays un-rotated).  ``interleaved``: the RoPE layout of the query-side
    rotations (kc is rotated the same way by the caller).  Returns o:
    [U, Lq, G, D] fp64.
    """
    c = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    kc, vc, q, kq, vq = c(kc), c(vc), c(q), c(kq), c(vq)
    U, P, D = kc.shape
    _, Lq, G, _ = q.shape
    o = np.zeros((U, Lq, G, D), np.float64)
    rc = _load().kvo_query_attention_units(U, P, Lq, G, D, float(theta), int(bool(interleaved)),
                                           float(scale),
                                           _ptr(kc), _ptr(vc), _ptr(q), _ptr(kq), _ptr(vq),
                                           _ptr(o))
    if rc != 0:
        raise MemoryError("oracle attention ran out of memory")
    return o
