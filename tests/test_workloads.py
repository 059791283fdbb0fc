"""Workload recipes and the byte / flop model behind the rooflines."""
import numpy as np
import pytest

from rag_precomputed_kv_gb300 import workloads as W
from test_oracle_pins import read_golden


def test_chunk_kv_bytes_match_pages():
    g = read_golden("coinrag_chunk_kv_bytes.txt")
    cfg = W.CONFIGS[2]
    assert (cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, cfg.chunk_len) == (
        g["qwen2_layers"], g["qwen2_kv_heads"], g["qwen2_head_dim"], g["chunk_tokens"])
    chunk = cfg.chunk_len * cfg.kv_bytes_per_token()
    assert abs(chunk / 2**20 - g["chunk_bytes_approx_mb"]) < 0.5        # "about 28 MB"
    l32 = W.dataclasses.replace(cfg, n_layers=g["turborag_layers"])
    assert abs(l32.kv_bytes_per_token() / 1000 - g["token_bytes_approx_kb"]) < 1  # "about 65 KB"


@pytest.mark.parametrize("cid", sorted(W.CONFIGS))
def test_span_draws_valid_and_deterministic(cid):
    cfg = W.CONFIGS[cid]
    a, b = W.draw_spans(cfg), W.draw_spans(cfg)
    assert len(a) == cfg.batch
    for ra, rb in zip(a, b):
        assert np.array_equal(ra.spans, rb.spans)
        sp = ra.spans
        local = (sp[:, 0] & W.LOCAL_FLAG) != 0
        assert np.all(sp[:, 1] >= 0) and np.all(sp[:, 2] > sp[:, 1])
        assert np.all(sp[~local, 2] <= cfg.chunk_len)
        assert np.all(sp[~local, 0] < cfg.pool_entries)
        if cfg.prompt_len:
            assert tuple(sp[0]) == (cfg.prompt_id, 0, cfg.prompt_len)
        body = sp[~local][1 if cfg.prompt_len else 0:]
        if cfg.spans in ("random", "one-per-chunk"):
            lens = body[:, 2] - body[:, 1]
            assert lens.min() >= cfg.span_min and lens.max() <= cfg.span_max
            assert len(body) == cfg.k_spans
            assert len(np.unique(body[:, 0])) <= cfg.k_chunks
        if cfg.spans == "one-per-chunk":
            assert len(np.unique(body[:, 0])) == cfg.k_chunks


def test_prefix_lengths_of_fixed_configs():
    assert W.draw_spans(W.CONFIGS[2])[0].prefix_len == 32 + 5 * 512
    for r in W.draw_spans(W.CONFIGS[4]):
        assert r.prefix_len == 16 * 2048 + 15 * 32          # 33,248
        assert r.local_len == 15 * 32


def test_roofline_numerators():
    cfg = W.CONFIGS[2]
    reqs = W.draw_spans(cfg)
    assert W.assemble_bytes(cfg, reqs) == 2 * 2592 * 57344
    P, lq = 2592, 64
    assert W.attention_flops(cfg, reqs) == 4 * 128 * 28 * 28 * (lq * P + lq * (lq + 1) // 2)
    cfg5 = W.CONFIGS[5]
    assert abs(cfg5.pool_bytes() / 1e9 - 77.4) < 0.2
