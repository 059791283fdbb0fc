"""Benchmark of the precomputed-KV RAG hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic
requests: kvr_assemble (span gather + RoPE re-rotation + stitch) followed by
kvr_query_attention (query RoPE + K/V append + tcgen05 prefill attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl kvr|reference]

The default workload is the serving-scale pool (Qwen3-8B shape: 36 layers,
32 query / 8 KV heads, a resident pool of 1024 chunks x 512 tokens, ~77 GB;
batch 64 requests of 32 spans each after a 64-token system prompt, 128 query
tokens each): the configuration with the largest pool and batch.
Beside it, the line carries the per-request latency of the full-chunk-reuse
case (Qwen2-7B shape, five 512-token chunks after a 32-token system prompt,
64 query tokens, batch 1), timed over at least 200 single-request prefills.
Prints ONE JSON line (rank 0).  Timing: CUDA events on the
launching stream around every step, L2 flushed between steps outside the
events (256 MiB written, then 256 MiB of another buffer read, so that no step
pays for the flush's own dirty lines), a barrier and synchronize on both
sides of the timed region, max over ranks.  Each rank runs its own replica of the batch (the
path shards by request with no exchange), so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rag_precomputed_kv_gb300 import workloads as W  # noqa: E402

METRIC = "stitched KV tokens/s & HBM GB/s; query-attn TFLOP/s; per-request latency"
UNIT = "stitched tokens/s"
L2_FLUSH_BYTES = 256 << 20
HOST_POOL_MAX_BYTES = 8 << 30   # the pinned-host-pool leg copies the pool (K and V) to the host


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    if there is none for this workload or the kernel source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f).get(kernel) or []
    for rec in recs if isinstance(recs, list) else [recs]:
        if rec.get("workload") != workload:
            continue
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != rec["source_sha256_16"]:
                return None
        return rec["bytes_per_launch"]
    return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kvr_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------
class Workload:
    """A batch of requests with its pool, cache and query tensors on one GPU."""

    def __init__(self, cfg: W.Config, device, variant: str = "default"):
        """``variant``: the position / RoPE layout of the pool: "interleaved"
        RoPE pairs, keys "unrotated" (kept before RoPE, rotated at their
        stitched positions), or "composite" positions (the chunk-local ids
        kept, delta 0).  The N(0,1) keys stand for any of them: a rotated
        isotropic Gaussian pair is again one."""
        import torch
        from rag_precomputed_kv_gb300 import kvr
        self.cfg = cfg
        self.variant = variant
        self.composite = variant == "composite"
        self.reqs = W.draw_spans(cfg)
        self.t = W.make_tensors(cfg, self.reqs, device=device)
        self.locals = [(k, v) for k, v in zip(self.t.local_k, self.t.local_v) if k is not None]
        remap, n = {}, 0
        for b, k in enumerate(self.t.local_k):
            if k is not None:
                remap[b], n = n, n + 1
        spans = []
        for r in self.reqs:
            sp = r.spans.copy()
            loc = (sp[:, 0] & W.LOCAL_FLAG) != 0
            for i in np.nonzero(loc)[0]:
                sp[i, 0] = W.LOCAL_FLAG | remap[int(sp[i, 0] & ~W.LOCAL_FLAG)]
            spans.append(sp)
        self.spans = np.concatenate(spans)
        self.span_offsets = np.concatenate([[0], np.cumsum([len(s) for s in spans])]).astype(np.int32)
        self.prefix = np.array([r.prefix_len for r in self.reqs], np.int64)
        lq = cfg.query_len
        # each cache block: prefix + query rows + one row for a decode step
        self.cache_offsets = np.concatenate([[0], np.cumsum(self.prefix + lq + 1)]).astype(np.int64)
        self.q_offsets = (np.arange(len(self.reqs) + 1) * lq).astype(np.int32)
        rows = int(self.cache_offsets[-1]) * cfg.n_layers * cfg.n_kv_heads
        self.cache_k = torch.empty((rows, cfg.head_dim), dtype=self.t.pool_k.dtype, device=device)
        self.cache_v = torch.empty_like(self.cache_k)
        self.out = torch.empty_like(self.t.q)
        self.pool = kvr.Pool(self.t.pool_k, self.t.pool_v, cfg.n_q_heads, cfg.rope_theta,
                             keys_unrotated=variant == "unrotated", rope_interleaved=variant == "interleaved")
        self.plen = self.prefix.astype(np.int32)

    def step(self, q=None, kq=None, vq=None, out=None, skip_prefix_cache=False):
        """One prefill of the whole batch: a single kvr_prefill call."""
        self.pool.prefill(self.span_offsets, self.spans, self.cache_offsets, self.cache_k,
                          self.cache_v, self.q_offsets, self.t.q if q is None else q,
                          self.t.kq if kq is None else kq, self.t.vq if vq is None else vq,
                          self.out if out is None else out, locals_=self.locals,
                          composite=self.composite, skip_prefix_cache=skip_prefix_cache)


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def asm_bytes_of(cfg, wl) -> int:
    """Algorithmic bytes of one stitch: every stitched K and V row read once
    and written once."""
    return W.assemble_bytes(cfg, wl.reqs)


def job_throughput(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / max_over_ranks(seconds, world)


class L2Flush:
    """Empties the L2 of everything a step could reuse: writes a buffer twice
    the L2's size, then reads another one, so that the write's dirty lines are
    written back here and not during the next timed step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.sink)


def workload_config(args) -> W.Config:
    """The configuration, with --layers / --batch (smaller cases of a workload
    for profiling) applied; the bench line's config shows them."""
    import dataclasses
    cfg = W.CONFIGS[args.config]
    if args.layers:
        cfg = dataclasses.replace(cfg, n_layers=args.layers)
    if args.batch:
        cfg = dataclasses.replace(cfg, batch=args.batch)
    return cfg


def decode_timing(wl, cfg, dev, steps, warmup, flush):
    """A decode step after the prefill: a query token per request at row (and
    position) P_b + Lq, attending to rows 0..P_b + Lq; one kvr_query_attention
    call.  Timed two ways: `us_per_step` over consecutive steps (a decode
    loop: the host enqueues ahead, each step reads every cache block, and the
    step's K/V bytes exceed the L2 on every workload here), and `us_isolated`
    for one call after an L2 flush, launch latency included."""
    import torch
    stream = torch.cuda.current_stream()
    B = len(wl.reqs)
    gdec = torch.Generator(device=dev)
    gdec.manual_seed(cfg.seed + 7)
    L, Hq, Hkv, Dh = cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    q1 = torch.randn((L, B, Hq, Dh), generator=gdec, device=dev).to(wl.t.q.dtype)
    k1 = torch.randn((L, B, Hkv, Dh), generator=gdec, device=dev).to(wl.t.q.dtype)
    v1 = torch.randn((L, B, Hkv, Dh), generator=gdec, device=dev).to(wl.t.q.dtype)
    o1 = torch.empty_like(q1)
    n_dec = (wl.prefix + cfg.query_len).astype(np.int32)
    q1_off = np.arange(B + 1, dtype=np.int32)

    def step():
        wl.pool.query_attention(wl.cache_offsets, n_dec, q1_off, q1, k1, v1, wl.cache_k, wl.cache_v, o1)

    wl.step()
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    n_d = max(20, min(steps, 500))
    # consecutive steps, enqueued while the GPU still runs a sleep kernel, so
    # that they run back to back: a Python call (marshalling + the library's
    # host work) takes about as long as a batch-1 step, and timed live the
    # loop would measure the host instead
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush()
    torch.cuda._sleep(DECODE_AHEAD_CYCLES)
    e0.record(stream)
    h0 = time.perf_counter()
    for _ in range(n_d):
        step()
    host_us = (time.perf_counter() - h0) / n_d * 1e6
    e1.record(stream)
    torch.cuda.synchronize()
    loop_ms = e0.elapsed_time(e1) / n_d
    # isolated calls
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_d)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_d)]
    for k in range(n_d):
        flush()
        d0[k].record(stream)
        step()
        d1[k].record(stream)
    torch.cuda.synchronize()
    wl.pool.check()
    iso_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(d0, d1))
    elt = 2 if cfg.dtype == "bf16" else 4
    dec_bytes = int((n_dec.astype(np.int64) + 1).sum()) * L * Hkv * Dh * elt * 2
    hbm = peaks()["hbm_gbs"]
    return {"workload": cfg.name, "us_per_step": round(loop_ms * 1e3, 2), "steps": n_d, "kv_bytes": dec_bytes,
            "host_us_per_call": round(host_us, 2),
            "gbs": round(dec_bytes / (loop_ms * 1e-3) / 1e9, 1),
            "frac_hbm": round(dec_bytes / (loop_ms * 1e-3) / 1e9 / hbm, 4),
            "us_isolated": round(iso_ms * 1e3, 2),
            "frac_hbm_isolated": round(dec_bytes / (iso_ms * 1e-3) / 1e9 / hbm, 4),
            "what": "kvr_query_attention with one token per request (append at P_b + Lq, attend to all rows); "
                    "bytes = K and V rows read once; us_per_step: consecutive steps on the device, enqueued ahead "
                    "(no flush between them: the step reads more than the L2 holds); host_us_per_call: the Python "
                    "call that enqueues one step; us_isolated: one call after an L2 flush"}


def host_pool_timing(wl, cfg, steps, warmup, flush):
    """The same batch from a copy of the pool in pinned host memory (the GPU
    reads it over the CPU-GPU link through its unified address): the stitch
    alone (kvr_assemble), the query attention alone (kvr_query_attention, on
    the stitched cache), and kvr_prefill, which stitches by layer groups on a
    second stream so that each group's attention overlaps the next group's
    stitch.  Skipped for pools above HOST_POOL_MAX_BYTES."""
    import torch
    from rag_precomputed_kv_gb300 import kvr as K
    pool_bytes = 2 * wl.t.pool_k.numel() * wl.t.pool_k.element_size()
    if pool_bytes > HOST_POOL_MAX_BYTES:
        return {"skipped": f"pool of {pool_bytes / 2**30:.1f} GiB: not copied to pinned host memory "
                           f"(limit {HOST_POOL_MAX_BYTES / 2**30:.0f} GiB)"}
    try:
        hk, hv = wl.t.pool_k.cpu().pin_memory(), wl.t.pool_v.cpu().pin_memory()
    except RuntimeError as e:
        return {"skipped": f"pinned host copy failed: {e}"}
    stream = torch.cuda.current_stream()
    hp = K.Pool(hk, hv, cfg.n_q_heads, cfg.rope_theta, keys_unrotated=wl.variant == "unrotated",
                rope_interleaved=wl.variant == "interleaved")
    n_h = max(5, min(steps, 100))

    def timed(fn):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_h)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_h)]
        for k in range(n_h):
            flush()
            e0[k].record(stream)
            fn()
            e1[k].record(stream)
        torch.cuda.synchronize()
        hp.check()
        return statistics.mean(a.elapsed_time(b) for a, b in zip(e0, e1))

    asm = lambda: hp.assemble(wl.span_offsets, wl.spans, wl.cache_offsets, wl.cache_k, wl.cache_v,
                              locals_=wl.locals, composite=wl.composite)
    att = lambda: hp.query_attention(wl.cache_offsets, wl.plen, wl.q_offsets, wl.t.q, wl.t.kq, wl.t.vq,
                                     wl.cache_k, wl.cache_v, wl.out)
    pre = lambda: hp.prefill(wl.span_offsets, wl.spans, wl.cache_offsets, wl.cache_k, wl.cache_v, wl.q_offsets,
                             wl.t.q, wl.t.kq, wl.t.vq, wl.out, locals_=wl.locals, composite=wl.composite)
    a_ms, q_ms, p_ms = timed(asm), timed(att), timed(pre)
    host_read = W.assemble_bytes(cfg, wl.reqs) // 2
    hp.close()
    return {"workload": cfg.name, "assemble_us": round(a_ms * 1e3, 2), "query_attention_us": round(q_ms * 1e3, 2),
            "serial_sum_us": round((a_ms + q_ms) * 1e3, 2), "prefill_us": round(p_ms * 1e3, 2), "steps": n_h,
            "host_read_gbs": round(host_read / (a_ms * 1e-3) / 1e9, 1),
            "what": "pool in pinned host memory, K/V rows read over the CPU-GPU link: kvr_assemble alone, "
                    "kvr_query_attention alone, and kvr_prefill (layer-group stitch on a second stream, each "
                    "group's attention beside the next group's stitch)"}


# the decode loop's head start: ~30 ms of GPU sleep while the host enqueues
# up to 500 steps
DECODE_AHEAD_CYCLES = 1 << 26

LATENCY_CONFIG = 2
LATENCY_REPS = 200


def latency_case(reps: int, warmup: int, dev, flush, variant: str = "default"):
    """Per-request latency: the full-chunk-reuse case (batch 1) as one
    kvr_prefill call, timed with CUDA events on its own over `reps` calls
    (L2 flushed before each), independent of the headline's step count.  The
    same calls are then repeated with the library's timing hook, for the
    stitch and attention kernels' own durations."""
    import torch
    cfg = W.CONFIGS[LATENCY_CONFIG]
    wl = Workload(cfg, dev, variant)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        wl.step()
    torch.cuda.synchronize()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    for k in range(reps):
        flush()
        e0[k].record(stream)
        wl.step()
        e1[k].record(stream)
    torch.cuda.synchronize()
    wl.pool.check()
    ms = sorted(a.elapsed_time(b) for a, b in zip(e0, e1))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(reps)]
    for e in [x for row in ev for x in row]:
        e.record(stream)
    torch.cuda.synchronize()
    for k in range(reps):
        flush()
        wl.pool.set_timing_events(ev[k])
        wl.step()
    torch.cuda.synchronize()
    wl.pool.set_timing_events(None)
    wl.pool.check()
    asm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.mean(e[4].elapsed_time(e[5]) for e in ev)
    pk = peaks()
    asm_gbs = W.assemble_bytes(cfg, wl.reqs) / (asm_ms * 1e-3) / 1e9
    att_tf = W.attention_flops(cfg, wl.reqs) / (att_ms * 1e-3) / 1e12
    res = {"workload": cfg.name, "reps": reps, "p50": round(ms[len(ms) // 2], 5),
           "p99": round(ms[min(len(ms) - 1, int(0.99 * len(ms)))], 5), "max": round(ms[-1], 5),
           "mean": round(statistics.mean(ms), 5),
           "attention": {"kernel": "k_attention_tc", "ms": round(att_ms, 5), "achieved": round(att_tf, 2),
                         "unit": "TFLOP/s", "frac": round(att_tf / pk["bf16_tflops"], 4),
                         "traffic": ncu_traffic("k_attention_tc", cfg.name)},
           "assemble": {"kernel": "k_assemble", "ms": round(asm_ms, 5), "achieved": round(asm_gbs, 1),
                        "unit": "GB/s", "frac": round(asm_gbs / pk["hbm_gbs"], 4),
                        "traffic": ncu_traffic("k_assemble", cfg.name)},
           "what": "one kvr_prefill call (stitch + query attention) for one request, device time per call, "
                   "L2 flushed before each; kernel durations from the timing hook (serialized)"}
    res["decode"] = decode_timing(wl, cfg, dev, reps, warmup, flush)
    res["host_pool"] = host_pool_timing(wl, cfg, reps, warmup, flush)
    wl.pool.close()
    return res


def run_kvr(args):
    import torch
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = workload_config(args)
    wl = Workload(cfg, dev, args.variant)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    from rag_precomputed_kv_gb300 import kvr as K

    for _ in range(args.warmup):
        flush()
        wl.step()
    torch.cuda.synchronize()
    wl.pool.check()

    # ---- timed region: device-resident inputs, one kvr_prefill per step ----
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in e0 + e1:   # create the CUDA events up front
        e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    host = 0.0
    for k in range(args.steps):
        flush()
        h0 = time.perf_counter()
        e0[k].record(stream)
        wl.step()
        e1[k].record(stream)
        host += time.perf_counter() - h0
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    wl.pool.check()
    step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)

    # ---- per-kernel durations: the library's timing hook records events
    # around each kernel (which serializes them), same steps otherwise ----
    n_kt = min(args.steps, 500)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_kt)]
    for e in [x for row in ev for x in row]:
        e.record(stream)
    torch.cuda.synchronize()
    for k in range(n_kt):
        flush()
        wl.pool.set_timing_events(ev[k])
        wl.step()
    torch.cuda.synchronize()
    wl.pool.set_timing_events(None)
    wl.pool.check()
    asm_ms = [e[0].elapsed_time(e[1]) for e in ev]
    app_ms = [e[2].elapsed_time(e[3]) for e in ev]
    att_ms = [e[4].elapsed_time(e[5]) for e in ev]
    ser_ms = [e[0].elapsed_time(e[5]) for e in ev]

    # ---- the same prefill with KVR_PREFILL_SKIP_PREFIX_CACHE (a keys-only
    # stitch; the attention gathers the prefix values from the pool), on the
    # tensor-core path ----
    gather = None
    if wl.pool.attention_path == K.PATH_TCGEN05:
        n_g = min(args.steps, 500)
        g0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_g)]
        g1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_g)]
        for _ in range(args.warmup):
            flush()
            wl.step(skip_prefix_cache=True)
        torch.cuda.synchronize()
        for k in range(n_g):
            flush()
            g0[k].record(stream)
            wl.step(skip_prefix_cache=True)
            g1[k].record(stream)
        torch.cuda.synchronize()
        wl.pool.check()
        g_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(g0, g1))
        # its kernels through the timing hook (serialized), as for the stitched step
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_g)]
        for e in [x for row in gev for x in row]:
            e.record(stream)
        torch.cuda.synchronize()
        for k in range(n_g):
            flush()
            wl.pool.set_timing_events(gev[k])
            wl.step(skip_prefix_cache=True)
        torch.cuda.synchronize()
        wl.pool.set_timing_events(None)
        wl.pool.check()
        gather = {"ms_per_step": round(g_ms, 5), "steps": n_g,
                  "value": round(int(wl.prefix.sum()) / (g_ms * 1e-3), 1), "unit": UNIT,
                  "kernel_ms": {
                      "stitch_keys": round(statistics.mean(e[0].elapsed_time(e[1]) for e in gev), 5),
                      "query_prologue": round(statistics.mean(e[2].elapsed_time(e[3]) for e in gev), 5),
                      "attention_values_gathered": round(statistics.mean(e[4].elapsed_time(e[5]) for e in gev), 5)},
                  "what": "kvr_prefill with KVR_PREFILL_SKIP_PREFIX_CACHE: a keys-only stitch, then the "
                          "attention reads the keys from the cache and gathers the prefix values from the "
                          "pool; the cache's prefix value rows are not written"}

    # ---- one decode step after the prefill ----
    decode = decode_timing(wl, cfg, dev, args.steps, args.warmup, flush)

    # ---- the prefill from a pool kept in pinned host memory ----
    host_pool = host_pool_timing(wl, cfg, args.steps, args.warmup, flush)

    # ---- end to end through the public API with host buffers ----
    # The batch is stitched with one kvr_assemble; its requests' query-side
    # work then runs in `e2e_chunks` consecutive groups, one kvr_query_attention
    # call each (as a server would split a large batch): each group's Q, K_q and
    # V_q go up on a copy stream (the copies start under the stitch, and a
    # group's copy overlaps the previous group's attention).  Each call's
    # output is written by the attention kernel straight into pinned host
    # memory (`--e2e-out host`, the default), or goes to device memory and down
    # on a second copy stream (`--e2e-out device`: slower, the two copy engines
    # share the link).  Every transfer of the step is inside its timed region
    # (the copy streams start after the step's start event).
    B_all = len(wl.reqs)
    n_ch = max(1, min(args.e2e_chunks, B_all))
    groups = [g for g in np.array_split(np.arange(B_all), n_ch) if len(g)]
    lq = cfg.query_len
    chunks = []
    for g in groups:
        b0, b1 = int(g[0]), int(g[-1]) + 1
        tsl = slice(b0 * lq, b1 * lq)
        ch = {"b0": b0, "b1": b1,
              "q_h": wl.t.q[:, tsl].contiguous().cpu().pin_memory(),
              "kq_h": wl.t.kq[:, tsl].contiguous().cpu().pin_memory(),
              "vq_h": wl.t.vq[:, tsl].contiguous().cpu().pin_memory(),
              "co": wl.cache_offsets[b0:b1 + 1].copy(),
              "qo": (np.arange(b1 - b0 + 1) * lq).astype(np.int32),
              "ev": torch.cuda.Event()}
        ch["q_d"], ch["kq_d"], ch["vq_d"] = (torch.empty(ch[k].shape, dtype=ch[k].dtype, device=dev)
                                             for k in ("q_h", "kq_h", "vq_h"))
        ch["out_h"] = torch.empty(ch["q_h"].shape, dtype=wl.out.dtype, pin_memory=True)
        if args.e2e_out == "device":
            ch["out_d"] = torch.empty(ch["q_h"].shape, dtype=wl.out.dtype, device=dev)
            ch["done"] = torch.cuda.Event()
        chunks.append(ch)
    h2d = sum(ch[k].numel() * ch[k].element_size() for ch in chunks for k in ("q_h", "kq_h", "vq_h"))
    d2h = sum(ch["out_h"].numel() * ch["out_h"].element_size() for ch in chunks)
    copy_s = torch.cuda.Stream()
    down_s = torch.cuda.Stream()

    def e2e_step():
        copy_s.wait_stream(stream)
        down_s.wait_stream(stream)
        with torch.cuda.stream(copy_s):
            for ch in chunks:
                for k in ("q", "kq", "vq"):
                    ch[k + "_d"].copy_(ch[k + "_h"], non_blocking=True)
                ch["ev"].record(copy_s)
        plen = wl.pool.assemble(wl.span_offsets, wl.spans, wl.cache_offsets, wl.cache_k, wl.cache_v,
                                locals_=wl.locals, composite=wl.composite)
        for ch in chunks:
            stream.wait_event(ch["ev"])
            wl.pool.query_attention(ch["co"], plen[ch["b0"]:ch["b1"]], ch["qo"], ch["q_d"], ch["kq_d"],
                                    ch["vq_d"], wl.cache_k, wl.cache_v, ch.get("out_d", ch["out_h"]))
            if "out_d" in ch:
                ch["done"].record(stream)
                down_s.wait_event(ch["done"])
                with torch.cuda.stream(down_s):
                    ch["out_h"].copy_(ch["out_d"], non_blocking=True)
        stream.wait_stream(copy_s)
        stream.wait_stream(down_s)

    for _ in range(args.warmup):
        flush()
        e2e_step()
    torch.cuda.synchronize()
    f0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    f1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush()
        f0[k].record(stream)
        e2e_step()
        f1[k].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(f0, f1)) / 1e3, world)
    # the same outputs as the device-resident steps, up to the rounding order of
    # the key halves merged for units that a smaller call splits (its last round)
    torch.testing.assert_close(torch.cat([ch["out_h"] for ch in chunks], dim=1).float(), wl.out.cpu().float(),
                               rtol=0, atol=2e-2)

    # ---- figures ----
    tokens_per_step = int(wl.prefix.sum())
    value = tokens_per_step * args.steps * world / total_s
    e2e_value = tokens_per_step * args.steps * world / e2e_s
    pk = peaks()
    asm_bytes = W.assemble_bytes(cfg, wl.reqs)
    att_flops = W.attention_flops(cfg, wl.reqs)
    asm_mean, att_mean, app_mean = (statistics.mean(x) for x in (asm_ms, att_ms, app_ms))
    asm_gbs = asm_bytes / (asm_mean * 1e-3) / 1e9
    att_tf = att_flops / (att_mean * 1e-3) / 1e12
    roof_asm = {"kernel": "k_assemble", "bound": "hbm", "achieved": round(asm_gbs, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(asm_gbs / pk["hbm_gbs"], 4),
                "traffic": None, "algorithmic_bytes": asm_bytes, "ms": round(asm_mean, 5),
                "peak_source": pk["source"]}
    roof_att = {"kernel": "k_attention_tc" if wl.pool.attention_path == K.PATH_TCGEN05 else "k_attention_simt",
                "bound": "tensor", "achieved": round(att_tf, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(att_tf / pk["bf16_tflops"], 4), "traffic": None,
                "algorithmic_flops": att_flops, "ms": round(att_mean, 5), "peak_source": pk["source"]}
    roof_asm["traffic"] = ncu_traffic("k_assemble", cfg.name)
    roof_att["traffic"] = ncu_traffic(roof_att["kernel"], cfg.name)
    dominant, other = (roof_asm, roof_att) if asm_mean >= att_mean else (roof_att, roof_asm)
    lat = sorted(step_ms)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded N(0,1) K/V/Q, random span draws; no datasets or weights)",
        "config": {"workload": cfg.name, "batch": cfg.batch, "layers": cfg.n_layers,
                   "q_heads": cfg.n_q_heads, "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
                   "chunk_len": cfg.chunk_len, "pool_entries": cfg.pool_entries,
                   "stitched_tokens_per_step": tokens_per_step, "query_tokens_per_request": cfg.query_len,
                   "l2": "flushed between steps outside the timed events: 256 MiB written, then 256 MiB "
                         "of another buffer read (the L2 holds no line of the step's data, and none dirty)",
                   "parallelism": f"request replicas x{world}", "variant": args.variant},
        "roofline": dominant, "roofline_other": other,
        "assemble_gbs": round(asm_gbs, 1), "attention_tflops": round(att_tf, 2),
        "append_ms": round(app_mean, 5),
        "kernel_timing": {"steps": n_kt, "ms_per_step_serialized": round(statistics.mean(ser_ms), 5),
                          "what": "per-kernel events from the library's timing hook, kernels serialized; "
                                  "ms_per_step above runs them overlapped (programmatic dependent launch)"},
        "host_ms_per_step": round(host * 1e3 / args.steps, 5),
        "step_ms": {"p50": round(lat[len(lat) // 2], 5), "max": round(lat[-1], 5),
                    "what": "one kvr_prefill call (stitch + query attention) per batch, device time"},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3 / args.steps, 5), "query_groups": len(chunks),
                "out": args.e2e_out,
                "what": "kvr_assemble for the batch, then one kvr_query_attention per group of requests; each "
                        "group's Q, K_q, V_q up from pinned host memory on a copy stream (under the stitch and the "
                        "previous group's attention); " + (
                            "each group's O into device memory, then down into pinned host memory on a second "
                            "copy stream (under the next group's work)" if args.e2e_out == "device" else
                            "O written by the attention kernel into pinned host memory") + "; per-step events"},
        "gpu_launches": 3 * args.steps,
        "skip_prefix_cache": gather,
        "decode": decode,
        "host_pool": host_pool,
        "clocks": clk,
    }
    if args.latency_reps > 0:
        res["latency_ms"] = latency_case(max(args.latency_reps, 1), args.warmup, dev, flush, args.variant)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.variant == "default":
        res["cpu_baseline"] = oracle_baseline(cfg, wl, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
class OracleSampler:
    """Times the fp64 oracle on bounded samples of the workload.

    A sample is the full assemble of U (layer, kv-head) units of request 0
    (U = the oracle's thread count) and its query attention restricted to the
    first lq_s query tokens (causal: those rows see exactly what they see in
    the full call).  The batch time is extrapolated linearly: assemble by
    stitched rows, attention by (query row, visible key) pairs.

    With a GPU workload ``wl`` the sample reads that workload's own tensors.
    Without one (the reference arm, which runs on the host alone) every
    (source, unit) row block and the sampled query rows are drawn N(0,1) on
    the host from generators seeded by (seed, source, unit): no pool is
    materialised, so a 77 GB workload samples as cheaply as a small one.
    """

    def __init__(self, cfg: W.Config, wl=None):
        import oracle
        oracle.build()
        self.oracle, self.cfg = oracle, cfg
        self.wl = wl
        if wl is not None:
            self.reqs = wl.reqs
            self.span_list = np.split(wl.spans, wl.span_offsets[1:-1])
        else:
            self.reqs = W.draw_spans(cfg)
            self.span_list = [r.spans for r in self.reqs]
        self.LH = cfg.n_layers * cfg.n_kv_heads
        self.threads = oracle.num_threads()
        self.set_units(min(self.LH, max(1, self.threads)))
        self.P0 = self.reqs[0].prefix_len
        self.tokens = int(sum(r.prefix_len for r in self.reqs))

    def _host_rows(self, tag, src, u, n, width):
        rng = np.random.default_rng([self.cfg.seed, tag, src & 0x7fffffff, u])
        x = rng.standard_normal((n, width))
        if self.cfg.dtype == "bf16":   # the values a bf16 input can hold
            import torch
            x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
        return x

    def set_units(self, n):
        """Sample the first n (layer, kv-head) units of request 0."""
        import torch
        cfg = self.cfg
        H, G, lq, D = cfg.n_kv_heads, cfg.group, cfg.query_len, cfg.head_dim
        self.units = list(range(n))
        self.sources = {}
        if self.wl is not None:
            t = self.wl.t
            to64 = lambda x: x.detach().to("cpu", torch.float64).numpy()
            li = torch.tensor([u // H for u in self.units])
            hi = torch.tensor([u % H for u in self.units])
            for s in np.unique(self.span_list[0][:, 0]):
                s = int(s)
                k, v = self.wl.locals[s & ~W.LOCAL_FLAG] if s & W.LOCAL_FLAG else (t.pool_k[s], t.pool_v[s])
                d = k.device
                self.sources[s] = (to64(k[li.to(d), hi.to(d)])[None], to64(v[li.to(d), hi.to(d)])[None])
            q, kq, vq = (to64(x[:, 0:lq]) for x in (t.q, t.kq, t.vq))
            self.qu = np.stack([q[u // H, :, (u % H) * G:(u % H + 1) * G] for u in self.units])
            self.kqu = np.stack([kq[u // H, :, u % H] for u in self.units])
            self.vqu = np.stack([vq[u // H, :, u % H] for u in self.units])
            return
        for s in np.unique(self.span_list[0][:, 0]):
            s = int(s)
            n_tok = self.reqs[0].local_len if s & W.LOCAL_FLAG else cfg.chunk_len
            k = np.stack([self._host_rows(0, s, u, n_tok, D) for u in self.units])[None]
            v = np.stack([self._host_rows(1, s, u, n_tok, D) for u in self.units])[None]
            self.sources[s] = (k, v)
        self.qu = np.stack([self._host_rows(2, 0, u, lq * G, D).reshape(lq, G, D) for u in self.units])
        self.kqu = np.stack([self._host_rows(3, 0, u, lq, D) for u in self.units])
        self.vqu = np.stack([self._host_rows(4, 0, u, lq, D) for u in self.units])

    @staticmethod
    def pairs(P, n):
        return n * (P + 1) + n * (n - 1) // 2

    def sample(self, lq_s):
        """(assemble seconds, attention seconds) of one sample."""
        o = self.oracle
        t0 = time.perf_counter()
        K, V, _ = o.assemble(self.sources, self.span_list[0], self.cfg.rope_theta)
        t1 = time.perf_counter()
        o.query_attention(K[0], V[0], self.qu[:, :lq_s], self.kqu[:, :lq_s], self.vqu[:, :lq_s],
                          self.cfg.rope_theta)
        return t1 - t0, time.perf_counter() - t1

    def batch_seconds(self, lq_s, t_asm, t_att):
        U, lq = len(self.units), self.cfg.query_len
        per_row = t_asm / max(1, self.P0) / U                  # one unit, one stitched row
        per_pair = t_att / self.pairs(self.P0, lq_s) / U       # one unit, one (row, key) pair
        total = 0.0
        for r in self.reqs:
            total += self.LH * (per_row * r.prefix_len + per_pair * self.pairs(r.prefix_len, lq))
        return total

    def choose_lq(self, budget_s):
        """Largest query-token count whose sample fits the budget."""
        t_asm, t_att1 = self.sample(1)
        per_pair = t_att1 / self.pairs(self.P0, 1)
        lq = self.cfg.query_len
        n = 1
        while n < lq and t_asm + per_pair * self.pairs(self.P0, n + 1) <= budget_s:
            n += 1
        return n

    def describe(self, lq_s):
        return (f"{len(self.units)} of {self.LH} (layer, kv-head) units of request 0: full assemble "
                f"({self.P0} stitched rows) + attention of the first {lq_s} of {self.cfg.query_len} query "
                f"tokens, fp64; extrapolated to the batch by rows and (row, key) pairs")


def oracle_baseline(cfg, wl, budget_s):
    smp = OracleSampler(cfg, wl)
    lq_s = smp.choose_lq(budget_s)
    t_asm, t_att = smp.sample(lq_s)
    if lq_s == cfg.query_len and t_asm + t_att < budget_s / 2 and len(smp.units) < smp.LH:
        # the whole query fits: widen the sample to more (layer, kv-head) units,
        # in multiples of the oracle's thread count, up to the budget
        per_set = max(t_asm + t_att, 1e-6)
        sets = max(1, min(-(-smp.LH // smp.threads), int(budget_s // per_set)))
        smp.set_units(min(smp.LH, sets * smp.threads))
        t_asm, t_att = smp.sample(lq_s)
    reps = 1
    if t_asm + t_att < budget_s / 2:
        # the sample is small against the budget: repeat it and average
        reps = max(1, min(8, int(budget_s // max(t_asm + t_att, 1e-6)) - 1))
        for _ in range(reps - 1):
            a_, b_ = smp.sample(lq_s)
            t_asm, t_att = t_asm + a_, t_att + b_
        t_asm, t_att = t_asm / reps, t_att / reps
    value = smp.tokens / smp.batch_seconds(lq_s, t_asm, t_att)
    return {"value": round(value, 2), "unit": UNIT, "cores": smp.threads, "kind": "oracle",
            "sample": smp.describe(lq_s) + f" ({reps} x {t_asm + t_att:.1f} s)"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = workload_config(args)
    smp = OracleSampler(cfg)
    per_step = max(0.02, args.ref_budget / (args.steps + args.warmup))
    lq_s = smp.choose_lq(per_step)
    if lq_s == cfg.query_len and len(smp.units) < smp.LH:
        # the whole query fits: widen the sample to more (layer, kv-head)
        # units, in multiples of the oracle's thread count, within the step's share
        t_asm, t_att = smp.sample(lq_s)
        sets = max(1, min(-(-smp.LH // smp.threads), int(0.8 * per_step // max(t_asm + t_att, 1e-6))))
        smp.set_units(min(smp.LH, sets * len(smp.units)))
    for _ in range(args.warmup):
        smp.sample(lq_s)
    spent, batch = [], []
    for _ in range(args.steps):
        t_asm, t_att = smp.sample(lq_s)
        spent.append(t_asm + t_att)
        batch.append(smp.batch_seconds(lq_s, t_asm, t_att))
    step_s = statistics.mean(spent)
    value = smp.tokens / statistics.mean(batch)
    sample = smp.describe(lq_s) + " per step"
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) K/V/Q drawn on the host per (source, unit), random span draws; "
                   "no datasets or weights)",
           "config": {"workload": cfg.name, "batch": cfg.batch, "stitched_tokens_per_step": smp.tokens,
                      "sample": sample,
                      "timing": "ms_per_step is the oracle's own time per step on that sample (what the run "
                                "spent); value is the whole batch's stitched tokens over the batch time "
                                "extrapolated from the sample, by stitched rows (assemble) and by (query row, "
                                "visible key) pairs (attention)",
                      "extrapolated_batch_ms": round(statistics.mean(batch) * 1e3, 3)},
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": smp.threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=sorted(W.CONFIGS))
    ap.add_argument("--e2e-out", default="host", choices=["device", "host"],
                    help="end-to-end step: output to device memory and copied down (device) or written "
                         "into pinned host memory by the attention kernel (host)")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="request groups of the end-to-end leg (one kvr_query_attention call each)")
    ap.add_argument("--latency-reps", type=int, default=LATENCY_REPS,
                    help="single-request prefills timed for the latency key (0: none)")
    ap.add_argument("--impl", default="kvr", choices=["kvr", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds of oracle work for the whole reference-arm run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    ap.add_argument("--variant", default="default", choices=["default", "interleaved", "unrotated", "composite"],
                    help="pool RoPE layout / positions (the oracle baseline is timed for the default only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvr(args)


if __name__ == "__main__":
    main()
