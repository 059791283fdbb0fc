"""Decode over the stitched cache (the step after prefill): each step is one
query token per request, appended at row n_b (position n_b) of its cache
block and attending to rows 0..n_b -- kvr_query_attention with one token per
request.  Several steps in a row after a kvr_prefill, checked against the
oracle, which builds its own cache (stitched prefix, query rows, earlier
decoded rows) from the same seeded inputs and never reads the GPU's.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from parity import Case, attn_within_tolerance, k_within_tolerance, to_np64
from rag_precomputed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STEPS = 3


def _run(cfg, reqs, sample_units=None, skip=(), il=False, turn=0, check=None, steps=STEPS, force_units=()):
    """`skip`: requests that take no token in the decode steps (q_len 0);
    `il`: a pool with interleaved RoPE pairs; `turn`: after the decode steps,
    a further query of that many tokens per request on the same cache (the
    next turn of a conversation); `check`: the requests compared with the
    oracle (default all; every request decodes either way)."""
    import torch
    case = Case(cfg, reqs=reqs, spare_rows=steps + 2 + turn, rope_interleaved=il)
    case.run(prefill=True)
    L, H, Hq, D = cfg.n_layers, cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim
    G, lq, B = Hq // H, cfg.query_len, len(case.reqs)
    dev = case.cache_k.device
    rng = np.random.default_rng(7)
    units = list(range(case.LH)) if sample_units is None else sorted(
        set(rng.choice(case.LH, size=sample_units, replace=False).tolist()) | set(force_units))
    checked = set(range(B) if check is None else check)
    li = [u // H for u in units]
    hi = [u % H for u in units]
    # the oracle's cache of every sampled unit: stitched prefix + query rows
    kc, vc = [], []
    for b in range(B):
        if b not in checked:   # never compared: a placeholder of the right length
            n_b = int(case.prefix[b]) + lq
            kc.append(np.zeros((0, n_b, D)))
            vc.append(np.zeros((0, n_b, D)))
            continue
        spans = case.spans[b]
        srcs = {int(s): case.source(int(s), units) for s in np.unique(spans[:, 0])}
        if srcs:
            K, V, pz = oracle.assemble(srcs, spans, cfg.rope_theta, interleaved=il)
            K, V = K[0], V[0]
        else:
            K = V = np.zeros((len(units), 0, D))
        P = K.shape[1]
        qo = int(case.q_offsets[b])
        kq = to_np64(case.t.kq[:, qo:qo + lq])
        vq = to_np64(case.t.vq[:, qo:qo + lq])
        kqu = np.stack([kq[l, :, h, :] for l, h in zip(li, hi)])
        vqu = np.stack([vq[l, :, h, :] for l, h in zip(li, hi)])
        kc.append(np.concatenate([K, oracle.rope(kqu, (P + np.arange(lq, dtype=np.float64))[None, :],
                                                  cfg.rope_theta, il)], axis=1))
        vc.append(np.concatenate([V, vqu], axis=1))
    g = torch.Generator(device=dev)
    g.manual_seed(99)
    dt = case.t.q.dtype
    act = [b for b in range(B) if b not in skip]
    tok = {b: i for i, b in enumerate(act)}
    qoffs = np.concatenate([[0], np.cumsum([0 if b in skip else 1 for b in range(B)])]).astype(np.int32)
    worst = (0.0, 0.0)
    for step in range(steps):
        n = np.array([kc[b].shape[1] for b in range(B)], np.int32)   # rows before this step
        T = len(act)
        q1 = torch.randn((L, T, Hq, D), generator=g, device=dev).to(dt)
        k1 = torch.randn((L, T, H, D), generator=g, device=dev).to(dt)
        v1 = torch.randn((L, T, H, D), generator=g, device=dev).to(dt)
        o1 = torch.full_like(q1, float("nan"))
        case.pool.query_attention(case.cache_offsets, n, qoffs, q1, k1, v1, case.cache_k, case.cache_v, o1)
        torch.cuda.synchronize()
        case.pool.check()
        q1n, k1n, v1n, o1n = (to_np64(x) for x in (q1, k1, v1, o1))
        for b in act:
            t = tok[b]
            if b not in checked:
                kc[b] = np.zeros((0, kc[b].shape[1] + 1, D))
                vc[b] = np.zeros((0, vc[b].shape[1] + 1, D))
                continue
            qu = np.stack([q1n[l, t, h * G:(h + 1) * G][None] for l, h in zip(li, hi)])   # [U, 1, G, D]
            ku = np.stack([k1n[l, t, h][None] for l, h in zip(li, hi)])                    # [U, 1, D]
            vu = np.stack([v1n[l, t, h][None] for l, h in zip(li, hi)])
            o_ref = oracle.query_attention(kc[b], vc[b], qu, ku, vu, cfg.rope_theta, interleaved=il)
            o_gpu = np.stack([o1n[l, t, h * G:(h + 1) * G][None] for l, h in zip(li, hi)])
            ok, mx, rel = attn_within_tolerance(o_gpu, o_ref, cfg.dtype)
            assert ok, (step, b, mx, rel)
            worst = (max(worst[0], mx), max(worst[1], rel))
            # the appended row: K rotated at n_b, V copied
            blk_k = to_np64(case.cache_block("k", b)[units])
            blk_v = to_np64(case.cache_block("v", b)[units])
            k_new = oracle.rope(ku, float(n[b]), cfg.rope_theta, il)
            okk, _ = k_within_tolerance(blk_k[:, n[b]:n[b] + 1], k_new, cfg.dtype, il)
            assert okk, (step, b)
            assert np.array_equal(blk_v[:, n[b]:n[b] + 1], vu), (step, b)
            kc[b] = np.concatenate([kc[b], k_new], axis=1)
            vc[b] = np.concatenate([vc[b], vu], axis=1)
    if turn:
        n = np.array([kc[b].shape[1] for b in range(B)], np.int32)
        qo2 = (np.arange(B + 1) * turn).astype(np.int32)
        q2 = torch.randn((L, B * turn, Hq, D), generator=g, device=dev).to(dt)
        k2 = torch.randn((L, B * turn, H, D), generator=g, device=dev).to(dt)
        v2 = torch.randn((L, B * turn, H, D), generator=g, device=dev).to(dt)
        o2 = torch.full_like(q2, float("nan"))
        case.pool.query_attention(case.cache_offsets, n, qo2, q2, k2, v2, case.cache_k, case.cache_v, o2)
        torch.cuda.synchronize()
        case.pool.check()
        q2n, k2n, v2n, o2n = (to_np64(x) for x in (q2, k2, v2, o2))
        for b in sorted(checked):
            sl = slice(b * turn, (b + 1) * turn)
            qu = np.stack([q2n[l, sl, h * G:(h + 1) * G] for l, h in zip(li, hi)])
            ku = np.stack([k2n[l, sl, h] for l, h in zip(li, hi)])
            vu = np.stack([v2n[l, sl, h] for l, h in zip(li, hi)])
            o_ref = oracle.query_attention(kc[b], vc[b], qu, ku, vu, cfg.rope_theta, interleaved=il)
            o_gpu = np.stack([o2n[l, sl, h * G:(h + 1) * G] for l, h in zip(li, hi)])
            ok, mx, rel = attn_within_tolerance(o_gpu, o_ref, cfg.dtype)
            assert ok, ("turn", b, mx, rel)
    return worst


EDGE = W.Config("edge", 2, 8, 2, 128, "bf16", 1e4, 4, 96, 5, 7, 1, 77, "random")


def test_decode_steps_after_prefill_bf16_tensor_cores():
    pid = EDGE.n_chunks
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in
            ([[pid, 0, 5], [0, 0, 96], [2, 10, 60]], [[1, 3, 90]], [])]
    cfg = dataclasses.replace(EDGE, batch=len(reqs), query_len=9)
    _run(cfg, reqs)


def test_decode_steps_fp32_cuda_cores():
    _run(W.CONFIGS[1], None)


def test_decode_steps_default_workload_sampled():
    _run(W.CONFIGS[2], None, sample_units=6)


def test_decode_step_serving_pool():
    """One decode step on the serving-scale workload (Qwen3-8B shape, 77 GB
    pool, 64 requests) after its prefill: every request decodes; requests
    0, 31 and 63 are compared, on 16 seeded units plus the last layer's
    first and last kv head."""
    c = W.CONFIGS[5]
    last = ((c.n_layers - 1) * c.n_kv_heads, c.n_layers * c.n_kv_heads - 1)
    _run(c, None, sample_units=16, check=[0, 31, 63], steps=1, force_units=last)


@pytest.mark.parametrize("variant", ["g1", "g16", "short_blocks_and_idle_requests", "interleaved_rope"])
def test_decode_kernel_edges(variant):
    """The streaming decode kernel: one and sixteen query heads per kv head,
    cache blocks shorter than one 128-key tile, requests that take no token
    in a step (their CTAs leave at once), interleaved RoPE pairs."""
    pid = EDGE.n_chunks
    lists = ([[pid, 0, 5], [0, 0, 96], [2, 10, 60]], [[1, 3, 90], [3, 0, 96]], [])
    skip, il = (), False
    if variant == "g1":
        cfg = dataclasses.replace(EDGE, n_q_heads=2, n_kv_heads=2, query_len=4)
    elif variant == "g16":
        cfg = dataclasses.replace(EDGE, n_q_heads=32, n_kv_heads=2, query_len=3, rope_theta=1e6)
    else:
        cfg = dataclasses.replace(EDGE, query_len=2)
        lists = ([[pid, 0, 5]], [[0, 10, 40]], [[1, 0, 96], [2, 0, 96]], [])
        skip = (1,)
    if variant == "interleaved_rope":
        cfg, il = dataclasses.replace(EDGE, n_q_heads=8, n_kv_heads=2, query_len=5), True
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in lists]
    _run(dataclasses.replace(cfg, batch=len(reqs)), reqs, skip=skip, il=il)


def test_decode_mixed_block_lengths():
    """One step over blocks of very different lengths: a long request (ten
    128-key tiles, its last one partial), a request of one partial tile, a
    request that takes no token, and seven query heads per kv head (the
    Qwen2-7B grouping, padded to sixteen MMA rows)."""
    pid = EDGE.n_chunks
    long_req = [[pid, 0, 5]] + [[c % 4, 0, 96] for c in range(12)]
    lists = (long_req, [[1, 3, 40]], [[2, 0, 96], [3, 10, 90]])
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in lists]
    cfg = dataclasses.replace(EDGE, n_q_heads=14, n_kv_heads=2, query_len=3, batch=len(reqs))
    _run(cfg, reqs, skip=(2,))


def test_next_turn_after_decode_steps():
    """Prefill, three decode steps, then a five-token query on the same cache
    (the next turn): the decode steps leave the V rows past their token as
    they are, and the query prologue pads them again for the tensor-core
    attention."""
    pid = EDGE.n_chunks
    reqs = [W.Request(np.asarray(r, np.int32).reshape(-1, 3), 0) for r in
            ([[pid, 0, 5], [0, 0, 96], [2, 10, 60]], [[1, 3, 90]], [[3, 0, 40]])]
    cfg = dataclasses.replace(EDGE, batch=len(reqs), query_len=9)
    _run(cfg, reqs, turn=5)
