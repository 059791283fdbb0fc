"""kvr_assemble_noalloc -- the assemble step for callers that cannot allocate.

Some callers cannot call cudaMalloc where they stitch a prefix (an engine
whose caching allocator already owns the free device memory, a request loop
that forbids allocations, a plug-in restricted to its host's allocator).
kvr_assemble_noalloc serves them with scratch in a fixed __device__ array.
These tests call it through the binding (argument marshalling over the C
ABI) and check that two calls in a row give exactly what kvr_assemble gives
(stitched K and V, position ids, source map, prefix lengths), and that it
refuses work beyond its fixed limits.

This file is collected last on purpose: it runs after every other test, and
also passes alone in a fresh process.
"""
import dataclasses

import numpy as np
import pytest
import torch

from parity import Case
from rag_precomputed_kv_gb300 import kvr
from rag_precomputed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _call(case, spans, span_offsets, ck, cv, pos, src, cache_offsets=None):
    """kvr_assemble_noalloc through the binding (the pool described on each
    call, with the same layout flags and positions as the Case's pool)."""
    return kvr.assemble_noalloc(case.t.pool_k, case.t.pool_v, case.cfg.n_q_heads, case.cfg.rope_theta,
                                span_offsets, spans,
                                case.cache_offsets if cache_offsets is None else cache_offsets, ck, cv,
                                locals_=case.locals, pos_ids=pos, src_map=src, composite=case.composite,
                                keys_unrotated=case.keys_unrotated, rope_interleaved=case.il)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


EDGE = W.Config("edge", 2, 8, 2, 128, "bf16", 1e4, 4, 96, 5, 7, 1, 77, "random")


def _past_4096():
    """Two requests, the first with a 4,805-row prefix: its positions cross
    2^12, where the RoPE table lookup changes form."""
    long_req = [[4, 0, 5]] + [[c % 4, 0, 96] for c in range(50)]
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in (long_req, [[1, 7, 60]])]
    return dataclasses.replace(EDGE, batch=len(reqs)), reqs


CASES = {
    "tiny-fp32": lambda: Case(W.CONFIGS[1], prerotate=False),
    "nuggets-b4": lambda: Case(W.with_batch(W.CONFIGS[3], 4), prerotate=False),
    "docs-inline-2-layers": lambda: Case(dataclasses.replace(W.CONFIGS[4], batch=1, n_layers=2, n_chunks=16),
                                         prerotate=False),
    # the pool's keys kept before RoPE: every token turned by its own position
    "keys-unrotated-past-4096": lambda: Case(*_past_4096()[:1], reqs=_past_4096()[1], prerotate=False,
                                             keys_unrotated=True),
    "keys-unrotated-with-locals": lambda: Case(dataclasses.replace(W.CONFIGS[4], batch=1, n_layers=2,
                                                                   n_chunks=16),
                                               prerotate=False, keys_unrotated=True),
    # adjacent-pair RoPE layout
    "interleaved-past-4096": lambda: Case(*_past_4096()[:1], reqs=_past_4096()[1], prerotate=False,
                                          rope_interleaved=True),
    "interleaved-fp32": lambda: Case(W.CONFIGS[1], prerotate=False, rope_interleaved=True),
    # composite positions: the chunk-local ids kept, no re-rotation
    "composite-nuggets-b2": lambda: Case(W.with_batch(W.CONFIGS[3], 2), prerotate=False, composite=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_assemble_on_two_calls(name):
    case = CASES[name]()
    case.run(attention=False)                       # kvr_assemble, the existing entry point
    ref = [case.cache_k.clone(), case.cache_v.clone(), case.pos_ids.clone(), case.src_map.clone()]
    spans = np.ascontiguousarray(np.concatenate(case.spans), np.int32)
    for call in range(2):
        ck = torch.full_like(case.cache_k, float("nan"))
        cv = torch.full_like(case.cache_v, float("nan"))
        pos = torch.full_like(case.pos_ids, -1)
        src = torch.full_like(case.src_map, -1)
        plen = _call(case, spans, case.span_offsets, ck, cv, pos, src)
        torch.cuda.synchronize()
        assert np.array_equal(plen, case.prefix), call
        assert torch.equal(_bits(ck), _bits(ref[0])), f"call {call}: K differs"
        assert torch.equal(_bits(cv), _bits(ref[1])), f"call {call}: V differs"
        assert torch.equal(pos, ref[2]) and torch.equal(src, ref[3]), f"call {call}: maps differ"


def test_noalloc_rejects_work_beyond_its_limits():
    case = Case(W.CONFIGS[1], prerotate=False)
    n = 4097                                        # one span more than the scratch holds
    spans = np.tile(np.array([[0, 0, 1]], np.int32), (n, 1))
    so = np.array([0, n], np.int32)
    co = np.array([0, n + 16], np.int64)
    ck = torch.empty((int(co[-1]) * case.LH, case.cfg.head_dim), dtype=case.cache_k.dtype, device="cuda")
    pos = torch.empty(n, dtype=torch.int32, device="cuda")
    src = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(kvr.KvrError) as ei:
        _call(case, spans, so, ck, ck, pos, src, cache_offsets=co)
    assert ei.value.status == 1                     # KVR_ERR_INVALID_ARG, before any GPU work
    assert "4096" in str(ei.value)                  # the reason names the limit
