"""The calls' asynchrony and allocation contract, and the device-side input
check.

After kvr_pool_reserve, calls within the reserved sizes enqueue their work
and return while the stream is still busy with earlier work: no allocation,
no free, no host wait (the header lists the only exceptions).  A NaN in a
query row is reported by kvr_check as KVR_ERR_DEVICE_CHECK, and the pool
stays usable.
"""
import dataclasses
import time

import numpy as np
import pytest
import torch

from parity import Case, run_parity_case
from rag_precomputed_kv_gb300 import kvr
from rag_precomputed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

EDGE = W.Config("edge", 2, 8, 2, 128, "bf16", 1e4, 4, 96, 5, 7, 1, 77, "random")
SLEEP_CYCLES = 1 << 30          # about half a second at the GB300's clock


def _query_inputs(case, lq, seed):
    """Query-side tensors for `lq` tokens per request (drawn up front, so no
    torch allocation happens while the calls are timed)."""
    cfg, B = case.cfg, len(case.reqs)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    T = B * lq
    q = torch.randn((cfg.n_layers, T, cfg.n_q_heads, cfg.head_dim), generator=g, device="cuda").bfloat16()
    kq = torch.randn((cfg.n_layers, T, cfg.n_kv_heads, cfg.head_dim), generator=g, device="cuda").bfloat16()
    vq = torch.randn_like(kq)
    out = torch.full_like(q, float("nan"))
    qo = (np.arange(B + 1) * lq).astype(np.int32)
    return q, kq, vq, out, qo


def test_reserved_calls_with_growing_query_enqueue_without_waiting():
    """Prefills of 4, 16, 64 and 160 query tokens per request (the query
    scratch grows 40x) over more than 64 spans (tables uploaded through the
    staging slots), all enqueued behind a half-second kernel: every call
    returns while that kernel still runs, and the results equal the same
    calls made on an idle stream."""
    rng = np.random.default_rng(3)
    lists = []
    for b in range(6):
        rows = [[EDGE.n_chunks, 0, 5]]
        for _ in range(14):
            c = int(rng.integers(0, EDGE.n_chunks))
            s0 = int(rng.integers(0, 80))
            rows.append([c, s0, s0 + int(rng.integers(1, 16))])
        lists.append(rows)
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in lists]
    lqs = (4, 16, 64, 160)
    cfg = dataclasses.replace(EDGE, batch=len(reqs), query_len=max(lqs))
    case = Case(cfg, reqs=reqs)
    spans = np.concatenate(case.spans)
    assert len(spans) > 64
    case.pool.reserve(max_batch=len(reqs), max_spans=len(spans), max_query_tokens=len(reqs) * max(lqs))
    assert case.pool.attention_path == kvr.PATH_TCGEN05
    inputs = [_query_inputs(case, lq, 10 + i) for i, lq in enumerate(lqs)]
    co = [np.concatenate([[0], np.cumsum(case.prefix + lq)]).astype(np.int64) for lq in lqs]
    # one call at the smallest size first: the kernels' modules load and their
    # launch attributes are set outside the timed calls
    q, kq, vq, out, qo = inputs[0]
    case.pool.prefill(case.span_offsets, spans, co[0], case.cache_k, case.cache_v, qo, q, kq, vq, out)
    torch.cuda.synchronize()
    case.pool.check()

    stream = torch.cuda.current_stream()
    torch.cuda._sleep(SLEEP_CYCLES)
    t0 = time.perf_counter()
    for (q, kq, vq, out, qo), c in zip(inputs, co):
        case.pool.prefill(case.span_offsets, spans, c, case.cache_k, case.cache_v, qo, q, kq, vq, out)
    host_s = time.perf_counter() - t0
    busy = not stream.query()
    torch.cuda.synchronize()
    case.pool.check()
    assert busy, "the stream went idle before the calls returned: a call waited for the GPU"
    assert host_s < 0.1, host_s
    got = [x[3].clone() for x in inputs]

    # the same calls on an idle stream, one at a time
    for (q, kq, vq, out, qo), c, g in zip(inputs, co, got):
        out.fill_(float("nan"))
        case.pool.prefill(case.span_offsets, spans, c, case.cache_k, case.cache_v, qo, q, kq, vq, out)
        torch.cuda.synchronize()
        case.pool.check()
        assert torch.equal(out.view(torch.int16), g.view(torch.int16))


def test_non_finite_query_is_reported_and_the_pool_stays_usable():
    """A NaN in one query head of one token: the tensor-core attention (and
    the decode kernel, for a one-token step) finds a row whose softmax
    denominator is not finite; kvr_check returns KVR_ERR_DEVICE_CHECK once,
    and the next call on the same pool passes parity."""
    pid = EDGE.n_chunks
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in
            ([[pid, 0, 5], [0, 3, 90]], [[1, 7, 60], [2, 0, 96]])]
    cfg = dataclasses.replace(EDGE, batch=len(reqs), query_len=9)
    case = Case(cfg, reqs=reqs, spare_rows=2)
    good = case.t.q.clone()
    case.t.q[1, 3, 5, 17] = float("nan")
    case.run(prefill=False, attention=False)
    plen = case.prefix.astype(np.int32)
    case.pool.query_attention(case.cache_offsets, plen, case.q_offsets, case.t.q, case.t.kq, case.t.vq,
                              case.cache_k, case.cache_v, case.out)
    with pytest.raises(kvr.KvrError) as e:
        case.pool.check()
    assert e.value.status == 6 and "finite" in str(e.value)
    case.pool.check()                                  # reported once
    # a decode step with a NaN in its query: the decode kernel reports it too
    n = (case.prefix + cfg.query_len).astype(np.int32)
    q1 = torch.randn((cfg.n_layers, 2, cfg.n_q_heads, cfg.head_dim), device="cuda").bfloat16()
    q1[0, 1, 0, 0] = float("inf")
    k1 = torch.randn((cfg.n_layers, 2, cfg.n_kv_heads, cfg.head_dim), device="cuda").bfloat16()
    v1, o1 = torch.randn_like(k1), torch.empty_like(q1)
    case.pool.query_attention(case.cache_offsets, n, np.arange(3, dtype=np.int32), q1, k1, v1,
                              case.cache_k, case.cache_v, o1)
    with pytest.raises(kvr.KvrError) as e:
        case.pool.check()
    assert e.value.status == 6
    case.t.q.copy_(good)
    res = run_parity_case(cfg=cfg, case=case, prefill=True)
    assert res["ok"], res
