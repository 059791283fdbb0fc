"""Parity harness: run the CUDA path through the C ABI and compare it with
the fp64 oracle on the same seeded inputs.

Tolerances (written here, used by every GPU parity test and by smoke()):
* position ids, source map, gathered V, appended V: bit-exact;
* re-rotated K (bf16): within 2 bf16 ulps of the exact value, the ulp taken
  at max(|k_ref|, 2^-14 * |pair|) -- a float rotation carries an absolute
  error proportional to the norm of the (x_i, x_{i+D/2}) pair, so an element
  that nearly cancels cannot be resolved below that floor;
* re-rotated K (fp32): |k - k_ref| <= 2^-20 * |pair|;
* attention output (bf16): max |o - o_ref| <= 2e-2 and
  sum|o - o_ref| / sum|o_ref| <= 5e-3; (fp32): 1e-4 and 1e-5.
"""
from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import oracle  # noqa: E402
from rag_precomputed_kv_gb300 import workloads as W  # noqa: E402

ATTN_TOL = {"bf16": (2e-2, 5e-3), "fp32": (1e-4, 1e-5)}


def to_np64(t):
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def pair_norm(x, interleaved=False):
    """Norm of the RoPE pair each element belongs to."""
    if interleaved:
        n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
        return np.repeat(n, 2, axis=-1)
    h = x.shape[-1] // 2
    n = np.sqrt(x[..., :h] ** 2 + x[..., h:] ** 2)
    return np.concatenate([n, n], axis=-1)


def k_within_tolerance(gpu, ref, dtype, interleaved=False):
    """Returns (ok, worst ratio of |err| to the allowed error)."""
    err = np.abs(gpu - ref)
    nrm = pair_norm(ref, interleaved)
    if dtype == "bf16":
        mag = np.maximum(np.abs(ref), 2.0 ** -14 * nrm)
        mag = np.where(mag > 0, mag, 2.0 ** -126)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        allowed = 2 * ulp
    else:
        allowed = np.maximum(2.0 ** -20 * nrm, 1e-30)
    ratio = float((err / allowed).max()) if err.size else 0.0
    return ratio <= 1.0, ratio


def attn_within_tolerance(gpu, ref, dtype):
    max_abs, mean_rel = ATTN_TOL[dtype]
    d = np.abs(gpu - ref)
    mx = float(d.max()) if d.size else 0.0
    rel = float(d.sum() / max(np.abs(ref).sum(), 1e-300)) if d.size else 0.0
    return (mx <= max_abs and rel <= mean_rel), mx, rel


class Case:
    """Inputs, layout and GPU results of one configuration."""

    def __init__(self, cfg: W.Config, device="cuda:0", prerotate=None, reqs=None, composite=False,
                 spare_rows=0, keys_unrotated=False, rope_interleaved=False):
        import torch
        from rag_precomputed_kv_gb300 import kvr
        self.cfg, self.device, self.composite = cfg, device, composite
        self.keys_unrotated = keys_unrotated   # pool keys kept before RoPE
        self.il = rope_interleaved             # RoPE pairs (x_2i, x_2i+1)
        self.reqs = reqs if reqs is not None else W.draw_spans(cfg)
        self.t = W.make_tensors(cfg, self.reqs, device=device)
        # explicit pre-rotation of the pool keys at chunk-local positions (the
        # offline forward pass of CoinRAG 2.1), done by the oracle in fp64
        if prerotate is None:
            prerotate = cfg.pool_bytes() < 2e9 and not keys_unrotated
        self.raw_pool_k = None
        if prerotate:
            raw = to_np64(self.t.pool_k)
            self.raw_pool_k = raw
            pos = np.arange(cfg.chunk_len, dtype=np.float64)[None, None, None, :]
            rot = oracle.rope(raw, np.broadcast_to(pos, raw.shape[:-1]), cfg.rope_theta, self.il)
            self.t.pool_k.copy_(torch.from_numpy(rot).to(self.t.pool_k.dtype))
        L, H, D = cfg.n_layers, cfg.n_kv_heads, cfg.head_dim
        self.LH = L * H
        # request-local sources: dense list, spans re-indexed
        self.locals, remap = [], {}
        for b, r in enumerate(self.reqs):
            if self.t.local_k[b] is not None:
                remap[b] = len(self.locals)
                self.locals.append((self.t.local_k[b], self.t.local_v[b]))
        spans = []
        for r in self.reqs:
            sp = r.spans.copy()
            loc = (sp[:, 0] & W.LOCAL_FLAG) != 0
            sp[loc, 0] = W.LOCAL_FLAG | np.array([remap[int(s & ~W.LOCAL_FLAG)] for s in sp[loc, 0]],
                                                 dtype=np.int64).astype(np.int32)
            spans.append(sp)
        self.spans = spans
        self.span_offsets = np.concatenate([[0], np.cumsum([len(s) for s in spans])]).astype(np.int32)
        self.prefix = np.array([r.prefix_len for r in self.reqs], np.int64)
        lq = cfg.query_len
        # cache blocks of P + Lq rows, plus `spare_rows` unused rows (left NaN)
        self.cache_offsets = np.concatenate([[0], np.cumsum(self.prefix + lq + spare_rows)]).astype(np.int64)
        self.q_offsets = (np.arange(len(self.reqs) + 1) * lq).astype(np.int32)
        rows = int(self.cache_offsets[-1]) * self.LH
        tdt = self.t.pool_k.dtype
        self.cache_k = torch.full((rows, D), float("nan"), dtype=tdt, device=device)
        self.cache_v = torch.full((rows, D), float("nan"), dtype=tdt, device=device)
        tot = int(self.prefix.sum())
        self.pos_ids = torch.full((max(tot, 1),), -1, dtype=torch.int32, device=device)
        self.src_map = torch.full((max(tot, 1), 2), -1, dtype=torch.int32, device=device)
        self.out = torch.full_like(self.t.q, float("nan"))
        self.pool = kvr.Pool(self.t.pool_k, self.t.pool_v, cfg.n_q_heads, cfg.rope_theta,
                             keys_unrotated=keys_unrotated, rope_interleaved=rope_interleaved)

    def run(self, attention=True, prefill=False, skip_prefix=False):
        """The hot path through the C ABI: kvr_assemble then
        kvr_query_attention, or (prefill=True) the single kvr_prefill call."""
        import torch
        if prefill:
            assert attention
            plen = self.pool.prefill(self.span_offsets, np.concatenate(self.spans), self.cache_offsets,
                                     self.cache_k, self.cache_v, self.q_offsets, self.t.q, self.t.kq,
                                     self.t.vq, self.out, locals_=self.locals, pos_ids=self.pos_ids,
                                     src_map=self.src_map, composite=self.composite,
                                     skip_prefix_cache=skip_prefix)
            assert np.array_equal(plen, self.prefix)
            torch.cuda.synchronize()
            self.pool.check()
            return
        plen = self.pool.assemble(self.span_offsets, np.concatenate(self.spans), self.cache_offsets,
                                  self.cache_k, self.cache_v, locals_=self.locals,
                                  pos_ids=self.pos_ids, src_map=self.src_map,
                                  composite=self.composite)
        assert np.array_equal(plen, self.prefix)
        if attention:
            self.pool.query_attention(self.cache_offsets, plen, self.q_offsets, self.t.q, self.t.kq,
                                      self.t.vq, self.cache_k, self.cache_v, self.out)
        torch.cuda.synchronize()
        self.pool.check()

    # ---- per-request views ----
    def cache_block(self, which, b):
        c = self.cache_k if which == "k" else self.cache_v
        r0, r1 = int(self.cache_offsets[b]), int(self.cache_offsets[b + 1])
        return c[r0 * self.LH: r1 * self.LH].view(self.LH, r1 - r0, -1)

    def source(self, src, units):
        """(k, v) of a source for the chosen (layer, kv-head) units, [1, U, n, D]."""
        import torch
        L, H = self.cfg.n_layers, self.cfg.n_kv_heads
        li = torch.tensor([u // H for u in units], device=self.device)
        hi = torch.tensor([u % H for u in units], device=self.device)
        if src & W.LOCAL_FLAG:
            k, v = self.locals[src & ~W.LOCAL_FLAG]
        else:
            k, v = self.t.pool_k[src], self.t.pool_v[src]
        return to_np64(k[li, hi])[None], to_np64(v[li, hi])[None]


def run_parity_case(cid=None, cfg=None, device="cuda:0", sample_units=None, requests=None,
                    attention=True, composite=False, seed_units=0, case=None, prefill=False,
                    skip_prefix=False, force_units=()):
    """Run one configuration and compare with the oracle; returns a summary
    dict with ``ok`` and the worst errors.  skip_prefix: kvr_prefill with
    KVR_PREFILL_SKIP_PREFIX_CACHE, whose cache prefix value rows must stay as
    they were (NaN), everything else compared as usual.  ``sample_units`` seeded
    (layer, kv-head) units are checked per request, plus ``force_units``
    (e.g. the last layer's)."""
    import torch
    cfg = cfg or W.CONFIGS[cid]
    case = case or Case(cfg, device=device, composite=composite)
    case.run(attention=attention, prefill=prefill, skip_prefix=skip_prefix)
    rng = np.random.default_rng(1234 + seed_units)
    req_ids = range(len(case.reqs)) if requests is None else requests
    L, H, Hq, D = cfg.n_layers, cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim
    G = Hq // H
    lq = cfg.query_len
    res = dict(ok=True, k_ratio=0.0, attn_max_abs=0.0, attn_mean_rel=0.0, units=0)
    pos_all = case.pos_ids.cpu().numpy()
    src_all = case.src_map.cpu().numpy()
    flat0 = np.concatenate([[0], np.cumsum(case.prefix)])
    for b in req_ids:
        units = list(range(case.LH)) if sample_units is None else sorted(
            set(rng.choice(case.LH, size=min(sample_units, case.LH), replace=False).tolist())
            | {int(u) % case.LH for u in force_units})
        spans = case.spans[b]
        srcs = {int(s): case.source(int(s), units) for s in np.unique(spans[:, 0])}
        if srcs:
            unrot = {s for s in srcs if not (s & W.LOCAL_FLAG)} if case.keys_unrotated else ()
            K_ref, V_ref, pz = oracle.assemble(srcs, spans, cfg.rope_theta, composite=composite,
                                               unrotated=unrot, interleaved=case.il)
        else:   # a request without any prefix
            K_ref = V_ref = np.zeros((1, len(units), 0, D))
            pz = oracle.positions(spans, 0, composite)
        P = pz.total
        # maps: bit-exact
        f0 = int(flat0[b])
        if not (np.array_equal(pos_all[f0:f0 + P], pz.pos) and
                np.array_equal(src_all[f0:f0 + P, 0], pz.src_id) and
                np.array_equal(src_all[f0:f0 + P, 1], pz.src_tok)):
            res["ok"] = False
            res["maps"] = f"request {b}: position / source map mismatch"
        ck = to_np64(case.cache_block("k", b)[units])
        cv = to_np64(case.cache_block("v", b)[units])
        if skip_prefix:
            # the attention gathers the prefix values from the pool: the cache's
            # prefix value rows stay as they were
            if not np.isnan(cv[:, :P]).all():
                res["ok"] = False
                res["prefix"] = f"request {b}: prefix value rows were written"
        elif not np.array_equal(cv[:, :P], V_ref[0]):
            res["ok"] = False
            res["v"] = f"request {b}: gathered V differs"
        okk, ratio = k_within_tolerance(ck[:, :P], K_ref[0], cfg.dtype, case.il)
        res["k_ratio"] = max(res["k_ratio"], ratio)
        res["ok"] &= okk
        if attention:
            qo = int(case.q_offsets[b])
            li = [u // H for u in units]
            hi = [u % H for u in units]
            q = to_np64(case.t.q[:, qo:qo + lq])           # [L, Lq, Hq, D]
            kq = to_np64(case.t.kq[:, qo:qo + lq])         # [L, Lq, H, D]
            vq = to_np64(case.t.vq[:, qo:qo + lq])
            qu = np.stack([q[l, :, h * G:(h + 1) * G, :] for l, h in zip(li, hi)])
            kqu = np.stack([kq[l, :, h, :] for l, h in zip(li, hi)])
            vqu = np.stack([vq[l, :, h, :] for l, h in zip(li, hi)])
            o_ref = oracle.query_attention(K_ref[0], V_ref[0], qu, kqu, vqu, cfg.rope_theta,
                                           interleaved=case.il)
            og = to_np64(case.out[:, qo:qo + lq])
            o_gpu = np.stack([og[l, :, h * G:(h + 1) * G, :] for l, h in zip(li, hi)])
            oka, mx, rel = attn_within_tolerance(o_gpu, o_ref, cfg.dtype)
            res["attn_max_abs"] = max(res["attn_max_abs"], mx)
            res["attn_mean_rel"] = max(res["attn_mean_rel"], rel)
            res["ok"] &= oka
            # appended query rows: K rotated at P + t, V copied
            kq_ref = oracle.rope(kqu, (P + np.arange(lq, dtype=np.float64))[None, :], cfg.rope_theta,
                                 case.il)
            okq, rq = k_within_tolerance(ck[:, P:P + lq], kq_ref, cfg.dtype, case.il)
            res["k_ratio"] = max(res["k_ratio"], rq)
            res["ok"] &= okq
            if not np.array_equal(cv[:, P:P + lq], vqu):
                res["ok"] = False
                res["vq"] = f"request {b}: appended V differs"
        res["units"] += len(units)
    torch.cuda.synchronize()
    return res
