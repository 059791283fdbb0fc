"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances are defined in ``parity.py``: bit-exact position ids, source map
and V rows; re-rotated K within 2 bf16 ulps; attention within max-abs 2e-2
and mean relative error 5e-3 (bf16).
"""
import dataclasses

import numpy as np
import pytest

from parity import Case, run_parity_case
from rag_precomputed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _ok(res):
    assert res["ok"], res
    return res


def test_config1_tiny_fp32_full():
    _ok(run_parity_case(1))


def test_config1_composite_positions():
    _ok(run_parity_case(1, composite=True))


def test_config2_whole_chunks_full():
    from rag_precomputed_kv_gb300 import kvr
    case = Case(W.CONFIGS[2])
    _ok(run_parity_case(cfg=W.CONFIGS[2], case=case))
    assert case.pool.attention_path == kvr.PATH_TCGEN05


def test_fp32_and_head_dim_64_use_cuda_cores():
    from rag_precomputed_kv_gb300 import kvr
    case = Case(W.CONFIGS[1])
    case.run()
    assert case.pool.attention_path == kvr.PATH_CUDA_CORES


def _last_layer(cid):
    """The first and last kv head of the last layer (units of the last
    (layer, kv-head) rows of every cache block)."""
    c = W.CONFIGS[cid]
    return ((c.n_layers - 1) * c.n_kv_heads, c.n_layers * c.n_kv_heads - 1)


def test_config3_nuggets_sampled_units():
    """Every request of the batch, 16 seeded (layer, kv-head) units each plus
    the last layer's first and last kv head."""
    res = _ok(run_parity_case(3, sample_units=16, force_units=_last_layer(3)))
    assert res["units"] >= 16 * 16


def _custom(cfg, span_lists, local_lens=None):
    reqs = []
    for i, rows in enumerate(span_lists):
        sp = np.asarray(rows, np.int32).reshape(-1, 3)
        reqs.append(W.Request(sp, (local_lens or {}).get(i, 0)))
    return dataclasses.replace(cfg, batch=len(reqs)), reqs


EDGE_BASE = W.Config("edge", 2, 8, 1, 128, "bf16", 1e4, 4, 96, 5, 7, 1, 77, "random")


@pytest.mark.parametrize("variant", ["g8_bf16_d128", "g1_bf16_d64", "g2_fp32_d128", "g4_bf16_d64"])
def test_edge_spans(variant):
    """Length-1 spans, spans ending at the chunk end, overlapping spans, empty
    spans, a request with no prefix at all, a prompt-only request, a query
    length that is not a multiple of any tile, several GQA group sizes."""
    base = {
        "g8_bf16_d128": EDGE_BASE,
        "g1_bf16_d64": dataclasses.replace(EDGE_BASE, n_layers=3, n_q_heads=3, n_kv_heads=3, head_dim=64,
                                           query_len=33, rope_theta=1e6),
        "g2_fp32_d128": dataclasses.replace(EDGE_BASE, dtype="fp32", n_q_heads=4, n_kv_heads=2, query_len=9),
        "g4_bf16_d64": dataclasses.replace(EDGE_BASE, n_q_heads=8, n_kv_heads=2, head_dim=64, query_len=130,
                                           rope_theta=5e5),
    }[variant]
    pid = base.n_chunks
    cfg, reqs = _custom(base, [
        [[pid, 0, 5], [0, 0, 1], [1, 95, 96], [2, 10, 50], [2, 30, 70], [3, 0, 96], [1, 5, 5]],
        [],
        [[pid, 0, 5]],
        [[3, 95, 96], [0, 17, 18], [1, 40, 41]],
    ])
    case = Case(cfg, reqs=reqs)
    _ok(run_parity_case(cfg=cfg, case=case))


def test_inline_local_sources():
    """Request-local (inline) token blocks interleaved between documents, as
    in the SemPIC hit path, sharing the pool re-rotation path."""
    base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=16)
    F = W.LOCAL_FLAG
    cfg, reqs = _custom(base, [
        [[0, 0, 96], [F | 0, 0, 8], [2, 0, 96], [F | 0, 8, 16], [1, 0, 96]],
        [[3, 0, 96], [F | 1, 0, 5], [0, 0, 96]],
    ], local_lens={0: 16, 1: 5})
    case = Case(cfg, reqs=reqs)
    _ok(run_parity_case(cfg=cfg, case=case))


def test_large_batch_uses_uploaded_tables():
    """More requests and spans than fit inside the kernel parameters: the span
    and request tables travel through the staging upload instead."""
    base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=3)
    rng = np.random.default_rng(5)
    lists = []
    for b in range(70):
        rows = []
        for _ in range(int(rng.integers(0, 3))):
            c = int(rng.integers(0, base.n_chunks))
            s0 = int(rng.integers(0, 90))
            rows.append([c, s0, s0 + int(rng.integers(1, 7))])
        lists.append(rows)
    cfg, reqs = _custom(base, lists)
    case = Case(cfg, reqs=reqs)
    _ok(run_parity_case(cfg=cfg, case=case, requests=[0, 1, 33, 68, 69]))


@pytest.mark.parametrize("spare", [1, 37, 200])
def test_cache_blocks_with_spare_rows(spare):
    """Cache blocks larger than prefix + query, their spare rows left NaN:
    masked keys must never pick up the garbage."""
    cfg = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, query_len=21)
    pid = cfg.n_chunks
    cfg, reqs = _custom(cfg, [[[pid, 0, 5], [0, 3, 50]], [[1, 0, 96], [2, 7, 9]], []])
    case = Case(cfg, reqs=reqs, spare_rows=spare)
    _ok(run_parity_case(cfg=cfg, case=case))


@pytest.mark.parametrize("cid", [2, 3])
def test_outputs_are_deterministic(cid):
    """Repeated calls give bit-identical caches and outputs (no result may
    depend on which CTA finishes first, e.g. in the split-KV merge)."""
    import torch
    cfg = W.CONFIGS[cid] if cid == 2 else W.with_batch(W.CONFIGS[3], 2)
    case = Case(cfg, prerotate=False)
    case.run()
    first = (case.out.clone(), case.cache_k.clone(), case.cache_v.clone())
    for _ in range(3):
        case.run()
        assert torch.equal(case.out.view(torch.int16), first[0].view(torch.int16))
        assert torch.equal(case.cache_k.view(torch.int16), first[1].view(torch.int16))
        assert torch.equal(case.cache_v.view(torch.int16), first[2].view(torch.int16))


def test_repeat_calls_reuse_staging():
    """More calls than staging slots on one pool give the same results."""
    case = Case(W.CONFIGS[1])
    first = None
    for _ in range(6):
        case.run()
        out = case.out.float().cpu()
        if first is None:
            first = out
        assert (out == first).all()
    _ok(run_parity_case(cfg=W.CONFIGS[1], case=case))


def _outputs(case):
    return [x.clone() for x in (case.out, case.cache_k, case.cache_v, case.pos_ids, case.src_map)]


def _reset(case):
    for x in (case.out, case.cache_k, case.cache_v):
        x.fill_(float("nan"))
    case.pos_ids.fill_(-1)
    case.src_map.fill_(-1)


def _same_bits(a, b):
    import torch
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


def _prefill_case(name):
    if name == "cfg2":
        return W.CONFIGS[2], None
    if name == "cfg1_fp32":
        return W.CONFIGS[1], None
    if name == "no_prefix":      # nothing to stitch: the query kernels run alone
        cfg = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=19)
        return _custom(cfg, [[], [[0, 4, 4]]])
    if name == "uploaded_tables":   # > 64 spans and requests: staged uploads on both halves
        base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=3)
        rng = np.random.default_rng(11)
        lists = [[[int(rng.integers(0, base.n_chunks)), 5, 5 + int(rng.integers(1, 9))]
                  for _ in range(int(rng.integers(1, 3)))] for _ in range(66)]
        return _custom(base, lists)
    raise ValueError(name)


@pytest.mark.parametrize("name", ["cfg2", "cfg1_fp32", "no_prefix", "uploaded_tables"])
def test_prefill_matches_oracle_and_the_two_calls(name):
    """kvr_prefill (the stitch and the query kernels launched back to back,
    overlapping) against the oracle, and bit for bit against kvr_assemble
    followed by kvr_query_attention."""
    cfg, reqs = _prefill_case(name)
    case = Case(cfg, reqs=reqs)
    few = None if len(case.reqs) <= 4 else [0, 1, len(case.reqs) // 2, len(case.reqs) - 1]
    _ok(run_parity_case(cfg=cfg, case=case, prefill=True, requests=few))
    got = _outputs(case)
    _reset(case)
    case.run()
    want = _outputs(case)
    for g, w in zip(got, want):
        assert _same_bits(g, w)
    # and once more through kvr_prefill after the two calls (scratch reuse)
    _reset(case)
    case.run(prefill=True)
    for g, w in zip(_outputs(case), want):
        assert _same_bits(g, w)


def test_config4_inline_docs_sampled():
    """All eight requests (33,248-row prefixes), 8 seeded units each plus
    the last layer's first and last kv head."""
    res = _ok(run_parity_case(4, sample_units=8, force_units=_last_layer(4)))
    assert res["units"] >= 8 * 8


def test_config5_serving_pool_sampled():
    """Eight requests spread over the batch of 64, the last one included
    (the shortest requests run in the attention's last, split round), 16
    seeded units each plus the last layer's first and last kv head."""
    reqs = [0, 9, 18, 27, 36, 45, 54, 63]
    res = _ok(run_parity_case(5, sample_units=16, requests=reqs, force_units=_last_layer(5)))
    assert res["units"] >= 8 * 16


@pytest.mark.parametrize("variant", ["fp32", "fp32_composite", "bf16_with_locals", "cfg2_prefill",
                                     "bf16_past_4096"])
def test_pool_keys_kept_before_rope(variant):
    """A pool registered with KVR_POOL_KEYS_UNROTATED: stitching applies RoPE
    at each token's position (request-local sources stay rotated at their
    local positions).  `bf16_past_4096`: a prefix of 4,805 rows, whose
    positions cross 2^12, where the RoPE table lookup changes form."""
    if variant == "bf16_past_4096":
        base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, query_len=9)
        long_req = [[4, 0, 5]] + [[c % 4, 0, 96] for c in range(50)]
        cfg, reqs = _custom(base, [long_req, [[1, 7, 60]]])
        composite = False
    elif variant.startswith("fp32"):
        cfg, reqs, composite = W.CONFIGS[1], None, variant.endswith("composite")
    elif variant == "bf16_with_locals":
        base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=11)
        F = W.LOCAL_FLAG
        cfg, reqs = _custom(base, [[[0, 3, 90], [F | 0, 0, 8], [2, 0, 40]], [[3, 10, 96], [1, 0, 5]]],
                            local_lens={0: 8})
        composite = False
    else:
        cfg, reqs, composite = W.CONFIGS[2], None, False
    case = Case(cfg, reqs=reqs, composite=composite, keys_unrotated=True)
    _ok(run_parity_case(cfg=cfg, case=case, composite=composite, prefill=variant == "cfg2_prefill"))


@pytest.mark.parametrize("variant", ["bf16_two_calls", "cfg2_prefill", "fp32_cuda_cores", "d64_cuda_cores",
                                     "unrotated_with_locals", "cfg2_gathering"])
def test_pool_with_interleaved_rope_pairs(variant):
    """A pool registered with KVR_POOL_ROPE_INTERLEAVED: every rotation
    (stitched keys, query keys, query heads; in the stitch kernel, the query
    prologue and the CUDA-core attention, and in the keys-only stitch of the
    skip-prefix-cache prefill) pairs (x_2i, x_2i+1)."""
    import torch
    pid = EDGE_BASE.n_chunks
    lists = [[[pid, 0, 5], [0, 0, 1], [1, 95, 96], [2, 10, 50], [2, 30, 70]], [],
             [[3, 0, 96], [1, 5, 40]]]
    kw, unrot, prefill, skip = {}, False, False, False
    if variant == "bf16_two_calls":
        cfg, reqs = _custom(dataclasses.replace(EDGE_BASE, query_len=29), lists)
    elif variant == "cfg2_prefill":
        cfg, reqs, prefill = W.CONFIGS[2], None, True
    elif variant == "fp32_cuda_cores":
        cfg, reqs = W.CONFIGS[1], None
    elif variant == "d64_cuda_cores":
        cfg, reqs = _custom(dataclasses.replace(EDGE_BASE, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                                query_len=17, rope_theta=5e5), lists)
    elif variant == "unrotated_with_locals":
        base = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, prompt_len=0, query_len=11)
        F = W.LOCAL_FLAG
        cfg, reqs = _custom(base, [[[0, 3, 90], [F | 0, 0, 8], [2, 0, 40]], [[3, 10, 96], [1, 0, 5]]],
                            local_lens={0: 8})
        unrot = True
    else:
        cfg, reqs, prefill, skip = W.CONFIGS[2], None, True, True
    case = Case(cfg, reqs=reqs, keys_unrotated=unrot, rope_interleaved=True)
    _ok(run_parity_case(cfg=cfg, case=case, prefill=prefill, skip_prefix=skip, **kw))
    if skip:    # keys from the same stitch kernel, values the pool's bytes: same bits
        got = case.out.clone()
        case.out.fill_(float("nan"))
        case.run(prefill=True)
        assert torch.equal(got.view(torch.int16), case.out.view(torch.int16))


@pytest.mark.parametrize("name", ["edge_2_layers", "cfg2_28_layers"])
def test_pool_in_pinned_host_memory(name):
    """A pool kept in pinned host memory (read by the stitch kernel through
    its unified address).  kvr_prefill then stitches it in layer groups on a
    second stream, each group's attention running beside the next group's
    stitch: the stitched cache is the device pool's bit for bit, the output
    matches the oracle (its rounding may differ from the device pool's run,
    whose attention splits its last round of units differently)."""
    import torch
    from parity import attn_within_tolerance, to_np64
    from rag_precomputed_kv_gb300 import kvr
    if name == "edge_2_layers":
        cfg = dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, query_len=13)
        pid = cfg.n_chunks
        cfg, reqs = _custom(cfg, [[[pid, 0, 5], [0, 3, 90], [2, 0, 96]], [[1, 7, 60], [3, 0, 96]]])
        sample = None
    else:
        cfg, reqs, sample = W.CONFIGS[2], None, 8
    case = Case(cfg, reqs=reqs)
    case.run(prefill=True)
    want = [x.clone() for x in (case.out, case.cache_k, case.cache_v)]
    hk, hv = case.t.pool_k.cpu().pin_memory(), case.t.pool_v.cpu().pin_memory()
    case.pool = kvr.Pool(hk, hv, cfg.n_q_heads, cfg.rope_theta)
    for x in (case.out, case.cache_k, case.cache_v):
        x.fill_(float("nan"))
    _ok(run_parity_case(cfg=cfg, case=case, prefill=True, sample_units=sample))
    for g_, w_ in zip((case.cache_k, case.cache_v), want[1:]):
        assert torch.equal(g_.view(torch.int16), w_.view(torch.int16))
    ok, mx, rel = attn_within_tolerance(to_np64(case.out), to_np64(want[0]), cfg.dtype)
    assert ok, (mx, rel)
    with pytest.raises(kvr.KvrError) as e:      # the values-gathering attention wants device memory
        case.run(prefill=True, skip_prefix=True)
    assert e.value.status == 3


def test_bounded_wait_timeout_is_reported_and_the_pool_stays_usable():
    """A kernel whose wait nothing completes gives up after its limit and
    records KVR_ERR_TIMEOUT; kvr_check reports it once, and the pool and the
    context then run the hot path as before."""
    from rag_precomputed_kv_gb300 import kvr
    cfg, reqs = _custom(dataclasses.replace(EDGE_BASE, query_len=9), [[[0, 0, 50], [1, 10, 96]], [[2, 0, 30]]])
    case = Case(cfg, reqs=reqs)
    case.pool.selftest_wait(20_000_000)   # 20 ms
    with pytest.raises(kvr.KvrError) as e:
        case.pool.check()
    assert e.value.status == 5            # KVR_ERR_TIMEOUT
    case.pool.check()                     # reported once
    _ok(run_parity_case(cfg=cfg, case=case, prefill=True))


def test_query_side_buffers_in_pinned_host_memory():
    """q, kq, vq and out in pinned host memory (read and written by the
    kernels through their unified addresses): the same bits as with device
    buffers, on the tensor-core (G = 2 and 4, one and several query tiles),
    decode and CUDA-core paths."""
    import torch
    for cfg, reqs in (_custom(dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, query_len=13),
                              [[[0, 3, 90], [2, 0, 96]], [[1, 7, 60]]]),
                      _custom(dataclasses.replace(EDGE_BASE, n_q_heads=8, n_kv_heads=2, query_len=70),
                              [[[0, 3, 90], [2, 0, 96], [1, 0, 96]], [[1, 7, 60]], []]),
                      _custom(dataclasses.replace(EDGE_BASE, n_q_heads=4, n_kv_heads=2, query_len=1),
                              [[[0, 3, 90]], [[1, 7, 60], [3, 0, 96]]]),
                      (W.CONFIGS[1], None)):
        case = Case(cfg, reqs=reqs)
        case.run(prefill=True)
        want_out, want_k = case.out.clone(), case.cache_k.clone()
        hq, hkq, hvq = (x.cpu().pin_memory() for x in (case.t.q, case.t.kq, case.t.vq))
        hout = torch.full(case.out.shape, float("nan"), dtype=case.out.dtype, pin_memory=True)
        case.cache_k.fill_(float("nan"))
        case.pool.prefill(case.span_offsets, np.concatenate(case.spans), case.cache_offsets, case.cache_k,
                          case.cache_v, case.q_offsets, hq, hkq, hvq, hout, locals_=case.locals)
        torch.cuda.synchronize()
        case.pool.check()
        bits = (lambda t: t.view(torch.int16)) if case.out.dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
        assert torch.equal(bits(hout), bits(want_out.cpu()))
        assert torch.equal(bits(case.cache_k), bits(want_k))
