"""GPU parity of kvr_prefill with KVR_PREFILL_SKIP_PREFIX_CACHE: a keys-only
stitch, then the attention reads the keys from the cache and gathers the
prefix values straight from the pool; the cache's prefix value rows are left
alone (NaN here), so a key tile that reaches past its cache block meets them.

Checked against the oracle (attention output, stitched keys, appended query
rows, position ids and source map) and, bit for bit, against the stitched
path: the keys come from the same stitch kernel, the values are the pool's
bytes, and the MMAs run in the same order, so the outputs must be identical.
"""
import dataclasses

import numpy as np
import pytest

from parity import Case, run_parity_case
from rag_precomputed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

EDGE = W.Config("edge", 2, 8, 2, 128, "bf16", 1e4, 4, 96, 5, 7, 1, 77, "random")


def _custom(cfg, span_lists, local_lens=None):
    local_lens = local_lens or {}
    reqs = [W.Request(np.asarray(rows, np.int32).reshape(-1, 3), local_lens.get(b, 0))
            for b, rows in enumerate(span_lists)]
    return dataclasses.replace(cfg, batch=len(reqs)), reqs


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _case(name):
    if name == "cfg2":
        return W.CONFIGS[2], None, {}
    if name == "cfg2_composite":
        return W.CONFIGS[2], None, {"composite": True}
    if name == "cfg3":
        return W.CONFIGS[3], None, {"sample_units": 6, "requests": [0, 7, 15]}
    if name == "cfg5":
        return W.CONFIGS[5], None, {"sample_units": 3, "requests": [0, 31, 63]}
    if name == "edges":
        # a request without prefix, a prompt-only one, length-1 spans, a span
        # ending at the chunk end, overlapping spans
        pid = EDGE.n_chunks
        cfg, reqs = _custom(dataclasses.replace(EDGE, query_len=21),
                            [[], [[pid, 0, 5]], [[0, 95, 96], [1, 0, 1], [2, 10, 96]],
                             [[3, 3, 50], [3, 20, 60], [pid, 0, 5]]])
        return cfg, reqs, {}
    if name == "mixed_long_short":
        # requests whose spans average 96 rows or more (value tiles through TMA
        # box loads) beside requests of short spans (through the gather warps),
        # in one batch; cache blocks with spare rows
        pid = EDGE.n_chunks
        cfg, reqs = _custom(dataclasses.replace(EDGE, query_len=21),
                            [[[0, 0, 96], [1, 0, 96], [2, 0, 96]], [[3, 5, 20], [0, 1, 9]],
                             [[pid, 0, 5], [1, 0, 96], [2, 0, 96], [3, 0, 96]], [[2, 0, 96], [3, 0, 96]],
                             [[1, 50, 96], [0, 0, 96]]])
        return cfg, reqs, {"spare_rows": 3}
    if name == "local_sources":
        # request-local sources (inline tokens) between pool spans
        F = W.LOCAL_FLAG
        cfg, reqs = _custom(dataclasses.replace(EDGE, prompt_len=0, query_len=13),
                            [[[0, 0, 96], [F | 0, 0, 8], [1, 0, 96], [2, 0, 96]],
                             [[3, 10, 40], [F | 1, 0, 8], [0, 5, 20]]], local_lens={0: 8, 1: 8})
        return cfg, reqs, {}
    if name == "docs_inline":
        # per-document caches with inline tokens between them (Llama-3.1-8B
        # shape, 16 documents, 2 layers)
        return dataclasses.replace(W.CONFIGS[4], batch=1, n_layers=2, n_chunks=16), None, {"sample_units": 4}
    if name == "many_requests":
        base = dataclasses.replace(EDGE, prompt_len=0, query_len=3)
        rng = np.random.default_rng(3)
        lists = [[[int(rng.integers(0, base.n_chunks)), 4, 4 + int(rng.integers(1, 70))]
                  for _ in range(int(rng.integers(1, 4)))] for _ in range(70)]
        cfg, reqs = _custom(base, lists)
        return cfg, reqs, {"requests": [0, 1, 35, 68, 69]}
    raise ValueError(name)


def _strided(case):
    """The same pool seen through views whose token axis has 8 rows of
    padding after each (entry, layer, kv-head) block: strides no longer those
    of a contiguous pool."""
    import torch
    from rag_precomputed_kv_gb300 import kvr

    def pad(x):
        E, L, H, T, D = x.shape
        big = torch.full((E, L, H, T + 8, D), float("nan"), dtype=x.dtype, device=x.device)
        big[:, :, :, :T] = x
        return big[:, :, :, :T]

    case.t.pool_k, case.t.pool_v = pad(case.t.pool_k), pad(case.t.pool_v)
    assert not case.t.pool_v.is_contiguous()
    case.pool.close()
    case.pool = kvr.Pool(case.t.pool_k, case.t.pool_v, case.cfg.n_q_heads, case.cfg.rope_theta)
    return case


@pytest.mark.parametrize("name", ["cfg2", "cfg2_composite", "cfg3", "cfg5", "edges", "mixed_long_short",
                                  "local_sources", "docs_inline", "strided_pool", "many_requests"])
def test_gathering_prefill_matches_oracle_and_stitched_path(name):
    import torch
    if name == "strided_pool":
        cfg, reqs, kw = _case("mixed_long_short")
    else:
        cfg, reqs, kw = _case(name)
    composite = kw.pop("composite", False)
    case = Case(cfg, reqs=reqs, composite=composite, spare_rows=kw.pop("spare_rows", 0))
    if name == "strided_pool":
        case = _strided(case)
    res = run_parity_case(cfg=cfg, case=case, prefill=True, skip_prefix=True, composite=composite, **kw)
    assert res["ok"], res
    got = [case.out.clone(), case.pos_ids.clone(), case.src_map.clone()]
    # the query rows of every block, appended by the query prologue
    qrows = []
    for b in range(len(case.reqs)):
        P, lq = int(case.prefix[b]), cfg.query_len
        qrows.append((case.cache_block("k", b)[:, P:P + lq].clone(), case.cache_block("v", b)[:, P:P + lq].clone()))
    for x in (case.out, case.cache_k, case.cache_v):
        x.fill_(float("nan"))
    case.pos_ids.fill_(-1)
    case.src_map.fill_(-1)
    case.run(prefill=True)
    want = [case.out, case.pos_ids, case.src_map]
    for g_, w_ in zip(got, want):
        assert torch.equal(_bits(g_), _bits(w_))
    for b, (k, v) in enumerate(qrows):
        P, lq = int(case.prefix[b]), cfg.query_len
        assert torch.equal(_bits(k), _bits(case.cache_block("k", b)[:, P:P + lq]))
        assert torch.equal(_bits(v), _bits(case.cache_block("v", b)[:, P:P + lq]))


def test_gathering_prefill_is_deterministic():
    import torch
    case = Case(W.CONFIGS[2], prerotate=False)
    case.run(prefill=True, skip_prefix=True)
    first = case.out.clone()
    for _ in range(3):
        case.run(prefill=True, skip_prefix=True)
        assert torch.equal(_bits(case.out), _bits(first))


def test_gathering_prefill_refuses_what_it_cannot_gather():
    """fp32 pools take the stitched path only."""
    from rag_precomputed_kv_gb300 import kvr
    case = Case(W.CONFIGS[1])
    with pytest.raises(kvr.KvrError) as e:
        case.run(prefill=True, skip_prefix=True)
    assert e.value.status == 3


def test_gathering_prefill_with_pool_keys_kept_before_rope():
    """With the pool's keys kept before RoPE the keys-only stitch turns each
    row by its position; output still bit-identical to the stitched path."""
    import torch
    cfg = W.CONFIGS[2]
    case = Case(cfg, keys_unrotated=True)
    res = run_parity_case(cfg=cfg, case=case, prefill=True, skip_prefix=True)
    assert res["ok"], res
    got = case.out.clone()
    case.out.fill_(float("nan"))
    case.run(prefill=True)
    assert torch.equal(_bits(got), _bits(case.out))
