"""Synthetic workloads: the five configurations, their seeded inputs and the
algorithmic byte / flop counts used for rooflines.

This module holds no arithmetic of the method itself (no positions, no
rotation, no attention).  It only draws random span lists and tensors from
fixed seeds and counts sizes, so both the CUDA path and the oracle can be fed
the same inputs from it.

Shapes follow the pages: 512-token chunks (CoinRAG blog section 3.1),
Qwen2-7B shape 28 layers / 4 KV heads / head dim 128 (CoinRAG blog 3.3),
nugget lengths of about a dozen words (CoinRAG Table 4), per-document caches
with request-side inline tokens (SemPIC page).  Retrieval is replaced by
uniform random draws; LongBench and the other datasets are not used.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

DTYPE_BYTES = {"bf16": 2, "fp32": 4}


@dataclass(frozen=True)
class Config:
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str            # "bf16" or "fp32"
    rope_theta: float
    n_chunks: int         # chunks in the resident pool (the prompt entry comes on top)
    chunk_len: int
    prompt_len: int       # system prompt tokens (pool entry n_chunks), 0 = none
    query_len: int
    batch: int
    seed: int
    spans: str            # span-drawing recipe, see draw_spans()
    k_chunks: int = 0     # distinct chunks per request
    k_spans: int = 0      # spans per request
    span_min: int = 0
    span_max: int = 0
    inline_len: int = 0   # inline tokens between documents (request-local source)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def elt(self) -> int:
        return DTYPE_BYTES[self.dtype]

    @property
    def pool_entries(self) -> int:
        return self.n_chunks + (1 if self.prompt_len > 0 else 0)

    @property
    def prompt_id(self) -> int:
        return self.n_chunks

    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token over all layers and KV heads."""
        return 2 * self.n_layers * self.n_kv_heads * self.head_dim * self.elt

    def pool_bytes(self) -> int:
        return self.pool_entries * self.chunk_len * self.kv_bytes_per_token()


CONFIGS = {
    1: Config("tiny-fp32", 1, 4, 2, 64, "fp32", 1e4, 3, 64, 8, 16, 1, 1001, "random",
              k_chunks=3, k_spans=5, span_min=4, span_max=16),
    2: Config("qwen2-7b-5-whole-chunks-b1", 28, 28, 4, 128, "bf16", 1e6, 5, 512, 32, 64, 1, 1002,
              "whole", k_chunks=5),
    3: Config("qwen2-7b-nuggets-b16", 28, 28, 4, 128, "bf16", 1e6, 256, 512, 32, 64, 16, 1003,
              "random", k_chunks=20, k_spans=40, span_min=8, span_max=48),
    4: Config("llama3.1-8b-16docs-inline-b8", 32, 32, 8, 128, "bf16", 5e5, 128, 2048, 0, 256, 8,
              1004, "docs", k_chunks=16, inline_len=32),
    5: Config("qwen3-8b-serving-pool-b64", 36, 32, 8, 128, "bf16", 1e6, 1024, 512, 64, 128, 64,
              1005, "one-per-chunk", k_chunks=32, k_spans=32, span_min=8, span_max=64),
}

LOCAL_FLAG = 1 << 30   # span source id flag: request-local source (inline tokens)


@dataclass
class Request:
    spans: np.ndarray           # int32 [k, 3]: (src, start, end), src may carry LOCAL_FLAG
    local_len: int = 0          # tokens in this request's local (inline) source

    @property
    def prefix_len(self) -> int:
        return int(np.maximum(self.spans[:, 2] - self.spans[:, 1], 0).sum())


def draw_spans(cfg: Config) -> List[Request]:
    """Seeded span lists for every request of ``cfg`` (numpy PCG64).

    * ``random``: ``k_chunks`` distinct chunks per request, ``k_spans`` spans
      each from a chunk drawn uniformly among them, length U[min, max], start
      U[0, chunk_len - length]; retrieval order = draw order.
    * ``one-per-chunk``: ``k_chunks`` distinct chunks, one span from each.
    * ``whole``: ``k_chunks`` distinct chunks, each whole, in a seeded order.
    * ``docs``: request b uses documents 16b..16b+15 whole, in a seeded order,
      with an ``inline_len``-token request-local block between consecutive docs.
    A ``prompt_len``-token system prompt span (pool entry ``n_chunks``) comes first.
    """
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    reqs = []
    for b in range(cfg.batch):
        rows = []
        if cfg.prompt_len > 0:
            rows.append((cfg.prompt_id, 0, cfg.prompt_len))
        local_len = 0
        if cfg.spans in ("random", "one-per-chunk"):
            chunks = rng.choice(cfg.n_chunks, size=cfg.k_chunks, replace=False)
            for i in range(cfg.k_spans):
                c = chunks[i] if cfg.spans == "one-per-chunk" else chunks[rng.integers(cfg.k_chunks)]
                ln = int(rng.integers(cfg.span_min, cfg.span_max + 1))
                st = int(rng.integers(0, cfg.chunk_len - ln + 1))
                rows.append((int(c), st, st + ln))
        elif cfg.spans == "whole":
            for c in rng.permutation(cfg.n_chunks)[: cfg.k_chunks]:
                rows.append((int(c), 0, cfg.chunk_len))
        elif cfg.spans == "docs":
            docs = b * cfg.k_chunks + rng.permutation(cfg.k_chunks)
            for i, d in enumerate(docs):
                if i > 0 and cfg.inline_len > 0:
                    s = (i - 1) * cfg.inline_len
                    rows.append((LOCAL_FLAG | b, s, s + cfg.inline_len))
                    local_len = s + cfg.inline_len
                rows.append((int(d), 0, cfg.chunk_len))
        else:
            raise ValueError(cfg.spans)
        reqs.append(Request(np.asarray(rows, dtype=np.int32).reshape(-1, 3), local_len))
    return reqs


# ----------------------------------------------------------------------------
# algorithmic work (roofline numerators)
# ----------------------------------------------------------------------------
def assemble_bytes(cfg: Config, reqs: List[Request]) -> int:
    """Read + write of every stitched K and V row."""
    return 2 * sum(r.prefix_len for r in reqs) * cfg.kv_bytes_per_token()


def append_bytes(cfg: Config, reqs: List[Request]) -> int:
    """Read + write of the query tokens' own K and V rows."""
    return 2 * len(reqs) * cfg.query_len * cfg.kv_bytes_per_token()


def attention_flops(cfg: Config, reqs: List[Request]) -> int:
    """QK^T and PV over the visible keys, causal tail counted exactly."""
    lq = cfg.query_len
    return sum(4 * cfg.head_dim * cfg.n_q_heads * cfg.n_layers *
               (lq * r.prefix_len + lq * (lq + 1) // 2) for r in reqs)


def attention_min_bytes(cfg: Config, reqs: List[Request]) -> int:
    """Cache K/V read once per (request, layer, kv-head), Q read, O written."""
    kv = sum(r.prefix_len + cfg.query_len for r in reqs) * cfg.kv_bytes_per_token()
    qo = 2 * len(reqs) * cfg.query_len * cfg.n_layers * cfg.n_q_heads * cfg.head_dim * cfg.elt
    return kv + qo


# ----------------------------------------------------------------------------
# tensors (torch; the CUDA path and the oracle receive the same values)
# ----------------------------------------------------------------------------
@dataclass
class Tensors:
    pool_k: "object"                 # [entries, L, H_kv, chunk_len, D]
    pool_v: "object"
    local_k: list = field(default_factory=list)   # per request [L, H_kv, local_len, D] or None
    local_v: list = field(default_factory=list)
    q: "object" = None               # [L, sum Lq, H_q, D]
    kq: "object" = None              # [L, sum Lq, H_kv, D]
    vq: "object" = None


def make_tensors(cfg: Config, reqs: List[Request], device="cuda", pool_chunks: Optional[int] = None):
    """Draw every input tensor N(0,1) from one generator seeded with the
    config's seed, in a fixed order: pool K, pool V, local K/V per request,
    Q, K_q, V_q.  Pool keys are treated as already rotated at their
    chunk-local positions (a rotated isotropic Gaussian pair is again an
    isotropic Gaussian pair, so the statistics are those of rotated keys).
    ``pool_chunks`` limits the pool size (tests of the tiny configurations).
    """
    import torch
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)
    n_ent = cfg.pool_entries if pool_chunks is None else pool_chunks
    shape = (n_ent, cfg.n_layers, cfg.n_kv_heads, cfg.chunk_len, cfg.head_dim)
    t = Tensors(torch.randn(shape, generator=g, device=device, dtype=tdt),
                torch.randn(shape, generator=g, device=device, dtype=tdt))
    for r in reqs:
        if r.local_len > 0:
            ls = (cfg.n_layers, cfg.n_kv_heads, r.local_len, cfg.head_dim)
            t.local_k.append(torch.randn(ls, generator=g, device=device, dtype=tdt))
            t.local_v.append(torch.randn(ls, generator=g, device=device, dtype=tdt))
        else:
            t.local_k.append(None)
            t.local_v.append(None)
    nq = cfg.query_len * len(reqs)
    t.q = torch.randn((cfg.n_layers, nq, cfg.n_q_heads, cfg.head_dim), generator=g, device=device, dtype=tdt)
    t.kq = torch.randn((cfg.n_layers, nq, cfg.n_kv_heads, cfg.head_dim), generator=g, device=device, dtype=tdt)
    t.vq = torch.randn((cfg.n_layers, nq, cfg.n_kv_heads, cfg.head_dim), generator=g, device=device, dtype=tdt)
    return t


def with_batch(cfg: Config, batch: int) -> Config:
    """Same configuration with another batch size (smaller parity cases)."""
    return dataclasses.replace(cfg, batch=batch)
