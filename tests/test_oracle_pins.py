"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here re-types the oracle's own formulas.  Each pin checks the oracle
against an independent fact:

* the worked position example of TurboRAG's Figure 5 (golden fixture);
* the span-position formula as the CoinRAG blog prints it (inclusive ends,
  section 2.3) and a brute-force concatenation of token lists;
* RoPE as complex multiplication (numpy complex128) in both pair layouts,
  closed forms on unit vectors, the adjacent layout as a relabelling of the
  half-split one, and the group properties the pages rely on (identity at 0,
  composition, relative-position invariance, re-rotating a cached key equals
  rotating the raw key at its target);
* attention against torch's scaled_dot_product_attention (a library routine)
  on the special case "one chunk at offset 0 plus the query" that reduces to
  plain causal attention, and closed forms (single visible key, zero query).

The pin functions are plain callables so that ``test_oracle_mutations.py``
can run them against copies of the oracle with planted mistakes.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            nums = [int(x) for x in rest]
            vals[key] = nums if len(nums) > 1 else nums[0]
    return vals


# ----------------------------------------------------------------------------
# independent RoPE: complex multiplication (library complex exp)
# ----------------------------------------------------------------------------
def rot_complex(x, shift, theta):
    """Rotate rows of x (fp64, [..., D]) by ``shift`` using complex numbers:
    pair (x_i, x_{i+D/2}) is z = x_i + 1j*x_{i+D/2}, multiplied by
    exp(1j * shift * theta**(-2i/D))."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    h = D // 2
    z = x[..., :h] + 1j * x[..., h:]
    freqs = theta ** (-2.0 * np.arange(h) / D)
    ang = np.asarray(shift, np.float64)[..., None] * freqs
    w = z * np.exp(1j * ang)
    return np.concatenate([w.real, w.imag], axis=-1)


# ----------------------------------------------------------------------------
# positions
# ----------------------------------------------------------------------------
def pin_fig5_worked_example():
    g = read_golden("turborag_fig5_positions.txt")
    l, n, lq = g["chunk_len"], g["n_chunks"], g["query_len"]
    spans = [[c, 0, l] for c in range(n)]
    comp = oracle.positions(spans, 0, composite=True)
    reo = oracle.positions(spans, 0, composite=False)
    # the query continues after the stitched prefix in both schemes
    q_ids = np.arange(reo.total, reo.total + lq)
    comp_1b = np.concatenate([comp.pos, q_ids]) + 1
    assert comp_1b.tolist() == list(g["composite_ids"])
    reo_1b = np.concatenate([reo.pos, q_ids]) + 1
    assert reo_1b.tolist() == list(range(1, n * l + lq + 1))   # contiguous
    # probe: query token at 13 vs token 3 (1-based) of chunk 2 (1-based)
    row = (g["probe_chunk"] - 1) * l + (g["probe_token"] - 1)
    qpos = g["probe_query_pos"]
    assert qpos - (comp.pos[row] + 1) == g["composite_distance"]
    assert qpos - (reo.pos[row] + 1) == g["reordered_distance"]


def pin_delta_formula_and_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(20):
        k = int(rng.integers(1, 12))
        p_len = int(rng.integers(0, 40))
        srcs = rng.integers(0, 5, k)
        lens = rng.integers(0, 20, k)
        starts = np.array([int(rng.integers(0, 64 - ln + 1)) for ln in lens])
        spans = np.stack([srcs, starts, starts + lens], 1)
        pz = oracle.positions(spans, p_len)
        # CoinRAG 2.3 as printed: Delta_i = |p| + sum_{j<i} (e_j - s_j + 1), with e_j the
        # inclusive last token; our spans are half-open, so e_j(incl) = end_j - 1.
        e_incl = spans[:, 2] - 1
        for i in range(k):
            expect = p_len + sum(int(e_incl[j] - spans[j, 1] + 1) for j in range(i))
            assert pz.target[i] == expect
            assert pz.delta[i] == expect - spans[i, 1]
        # brute force: concatenate the token lists of the spans in retrieval order
        toks = [(int(s), t) for s, a, b in spans for t in range(a, b)]
        assert pz.total == len(toks)
        assert pz.src_id.tolist() == [s for s, _ in toks]
        assert pz.src_tok.tolist() == [t for _, t in toks]
        assert pz.pos.tolist() == list(range(p_len, p_len + len(toks)))


def pin_composite_positions():
    spans = [[3, 5, 9], [1, 0, 2], [3, 30, 31]]
    pz = oracle.positions(spans, 100, composite=True)
    assert pz.delta.tolist() == [0, 0, 0]
    assert pz.pos.tolist() == [5, 6, 7, 8, 0, 1, 30]


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------
def pin_rope_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((17, 64))
    y = oracle.rope(x, 0.0, 1e4)
    assert np.array_equal(x, y)            # R(0) is exactly the identity


def pin_rope_vs_complex():
    rng = np.random.default_rng(2)
    for D, theta in ((64, 1e4), (128, 1e6), (128, 5e5), (8, 10.0)):
        x = rng.standard_normal((9, D))
        sh = rng.integers(-40000, 40000, 9).astype(np.float64)
        np.testing.assert_allclose(oracle.rope(x, sh, theta), rot_complex(x, sh, theta),
                                   rtol=0, atol=1e-9)


def pin_rope_closed_form():
    D, theta = 16, 100.0
    for i in range(D // 2):
        e = np.zeros(D)
        e[i] = 1.0
        y = oracle.rope(e, 1.0, theta)
        w = theta ** (-2.0 * i / D)
        expect = np.zeros(D)
        expect[i], expect[i + D // 2] = np.cos(w), np.sin(w)
        np.testing.assert_allclose(y, expect, atol=1e-15)
        e2 = np.zeros(D)
        e2[i + D // 2] = 1.0
        y2 = oracle.rope(e2, 1.0, theta)
        expect2 = np.zeros(D)
        expect2[i], expect2[i + D // 2] = -np.sin(w), np.cos(w)
        np.testing.assert_allclose(y2, expect2, atol=1e-15)


def pin_rope_composition_and_norm():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128))
    a, b = 1234.0, -517.0
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, 1e6), b, 1e6),
                               oracle.rope(x, a + b, 1e6), atol=1e-12)
    y = oracle.rope(x, 33247.0, 5e5)
    h = 64
    np.testing.assert_allclose(x[:, :h] ** 2 + x[:, h:] ** 2, y[:, :h] ** 2 + y[:, h:] ** 2,
                               rtol=1e-13)


def pin_rope_relative_position():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((2, 128))
    m, n, c = 700.0, 31.0, 2048.0
    d1 = oracle.rope(q, m, 1e6) @ oracle.rope(k, n, 1e6)
    d2 = oracle.rope(q, m + c, 1e6) @ oracle.rope(k, n + c, 1e6)
    assert abs(d1 - d2) < 1e-10


def rot_complex_adjacent(x, shift, theta):
    """The interleaved layout by complex numbers: pair (x_2i, x_2i+1) is
    z = x_2i + 1j*x_2i+1, multiplied by exp(1j * shift * theta**(-2i/D))."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    ang = np.asarray(shift, np.float64)[..., None] * theta ** (-2.0 * np.arange(D // 2) / D)
    w = z * np.exp(1j * ang)
    out = np.empty_like(x)
    out[..., 0::2] = w.real
    out[..., 1::2] = w.imag
    return out


def half_split_to_adjacent(D):
    """Index map: element 2i of the adjacent layout is element i of the
    half-split one, element 2i+1 is element i + D/2."""
    idx = np.empty(D, np.int64)
    idx[0::2] = np.arange(D // 2)
    idx[1::2] = np.arange(D // 2) + D // 2
    return idx


def pin_rope_interleaved():
    """Adjacent pairs: complex multiplication, unit-vector closed forms, and
    the same rotation as the half-split layout up to the index map above."""
    rng = np.random.default_rng(11)
    for D, theta in ((64, 1e4), (128, 1e6), (8, 10.0)):
        x = rng.standard_normal((7, D))
        sh = rng.integers(-40000, 40000, 7).astype(np.float64)
        y = oracle.rope(x, sh, theta, interleaved=True)
        np.testing.assert_allclose(y, rot_complex_adjacent(x, sh, theta), rtol=0, atol=1e-9)
        m = half_split_to_adjacent(D)
        np.testing.assert_allclose(y, oracle.rope(x[:, np.argsort(m)], sh, theta)[:, m],
                                   rtol=0, atol=1e-12)
    D, theta = 16, 100.0
    for i in range(D // 2):
        w = theta ** (-2.0 * i / D)
        e = np.zeros(D)
        e[2 * i] = 1.0
        expect = np.zeros(D)
        expect[2 * i], expect[2 * i + 1] = np.cos(w), np.sin(w)
        np.testing.assert_allclose(oracle.rope(e, 1.0, theta, interleaved=True), expect, atol=1e-15)


def pin_interleaved_layout_is_a_relabelling():
    """Attention scores are dot products, so storing every head in the
    adjacent layout (keys, queries, query keys relabelled by the same index
    map) and rotating with adjacent pairs gives the half-split result; the
    values keep their layout.  The stitch, likewise, is the half-split stitch
    relabelled."""
    rng = np.random.default_rng(12)
    U, P, Lq, G, D, theta = 3, 9, 5, 2, 16, 1e4
    m = half_split_to_adjacent(D)
    kc = rng.standard_normal((U, P, D))
    vc = rng.standard_normal((U, P, D))
    q = rng.standard_normal((U, Lq, G, D))
    kq = rng.standard_normal((U, Lq, D))
    vq = rng.standard_normal((U, Lq, D))
    ref = oracle.query_attention(kc, vc, q, kq, vq, theta)
    got = oracle.query_attention(kc[..., m], vc, q[..., m], kq[..., m], vq, theta, interleaved=True)
    np.testing.assert_allclose(got, ref, atol=1e-12)
    L, H, n = 2, 2, 12
    raw = {c: rng.standard_normal((L, H, n, D)) for c in (4, 7)}
    vals = {c: rng.standard_normal((L, H, n, D)) for c in raw}
    spans = [(7, 2, 9), (4, 0, 5), (7, 10, 12)]
    Kh, Vh, _ = oracle.assemble({c: (raw[c], vals[c]) for c in raw}, spans, theta, first_pos=3)
    Ki, Vi, _ = oracle.assemble({c: (raw[c][..., m], vals[c]) for c in raw}, spans, theta,
                                first_pos=3, interleaved=True)
    np.testing.assert_allclose(Ki, Kh[..., m], atol=1e-12)
    assert np.array_equal(Vi, Vh)


def pin_assemble_is_rope_at_target():
    """A span cached at chunk-local positions and re-rotated equals the raw key
    rotated at its target position; values are copied bit-exactly."""
    rng = np.random.default_rng(5)
    L, H, n, D, theta = 2, 3, 24, 32, 1e4
    raw = {c: rng.standard_normal((L, H, n, D)) for c in range(3)}
    vals = {c: rng.standard_normal((L, H, n, D)) for c in range(3)}
    local = np.arange(n, dtype=np.float64)
    cached = {c: rot_complex(raw[c], local[None, None, :], theta) for c in raw}
    spans = np.array([[2, 3, 11], [0, 0, 24], [2, 20, 21], [1, 7, 7], [1, 5, 9]])
    K, V, pz = oracle.assemble({c: (cached[c], vals[c]) for c in raw}, spans, theta, first_pos=6)
    row = 0
    for (c, s, e), tgt in zip(spans, pz.target):
        ln = e - s
        tpos = np.arange(tgt, tgt + ln, dtype=np.float64)
        np.testing.assert_allclose(K[:, :, row:row + ln], rot_complex(raw[c][:, :, s:e], tpos[None, None, :], theta),
                                   atol=1e-12)
        assert np.array_equal(V[:, :, row:row + ln], vals[c][:, :, s:e])
        row += ln
    assert row == pz.total


def pin_unrotated_sources_take_rope_at_their_positions():
    """Keys kept before RoPE and rotated at the stitched positions equal the
    same keys cached at chunk-local positions and re-rotated by delta (the
    rotation composes: R(target) k = R(delta) R(local) k), in both position
    schemes; values are untouched."""
    rng = np.random.default_rng(9)
    L, H, n, D, theta = 2, 2, 20, 16, 1e4
    raw = {c: rng.standard_normal((L, H, n, D)) for c in range(3)}
    vals = {c: rng.standard_normal((L, H, n, D)) for c in range(3)}
    local = np.arange(n, dtype=np.float64)
    cached = {c: rot_complex(raw[c], local[None, None, :], theta) for c in raw}
    spans = np.array([[1, 4, 12], [0, 0, 20], [2, 19, 20], [1, 0, 3]])
    for composite in (False, True):
        Kr, Vr, pz = oracle.assemble({c: (raw[c], vals[c]) for c in raw}, spans, theta, first_pos=3,
                                     composite=composite, unrotated=set(raw))
        Kc, Vc, _ = oracle.assemble({c: (cached[c], vals[c]) for c in raw}, spans, theta, first_pos=3,
                                    composite=composite)
        np.testing.assert_allclose(Kr, Kc, atol=1e-12)
        assert np.array_equal(Vr, Vc)
        # and, written out: each token's raw key rotated at its position id
        row = 0
        for c, s, e in spans:
            for t in range(s, e):
                np.testing.assert_allclose(Kr[:, :, row], rot_complex(raw[c][:, :, t], float(pz.pos[row]), theta),
                                           atol=1e-12)
                row += 1


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def _sdpa_causal(q, k, v):
    """torch's scaled_dot_product_attention, causal, fp64: [H, S, D] each."""
    with torch.no_grad():
        return torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
            is_causal=True)[0].numpy()


def pin_attention_single_chunk_is_causal_attention():
    """One chunk at offset 0 (delta 0) followed by the query reproduces plain
    causal attention over chunk + query (last Lq rows), with GQA heads."""
    rng = np.random.default_rng(6)
    for (Hkv, G, n, Lq, D, theta) in ((2, 2, 20, 6, 16, 1e4), (1, 3, 9, 5, 8, 100.0),
                                      (3, 1, 33, 4, 32, 1e6)):
        S = n + Lq
        raw_k = rng.standard_normal((Hkv, S, D))
        v = rng.standard_normal((Hkv, S, D))
        raw_q = rng.standard_normal((Hkv * G, S, D))
        pos = np.arange(S, dtype=np.float64)
        k_rot = rot_complex(raw_k, pos[None, :], theta)
        q_rot = rot_complex(raw_q, pos[None, :], theta)
        ref = _sdpa_causal(q_rot, np.repeat(k_rot, G, axis=0), np.repeat(v, G, axis=0))
        # oracle units = kv heads; its query heads h = u*G + g
        q_units = raw_q[:, n:, :].reshape(Hkv, G, Lq, D).transpose(0, 2, 1, 3)
        o = oracle.query_attention(k_rot[:, :n], v[:, :n], q_units, raw_k[:, n:], v[:, n:], theta)
        got = o.transpose(0, 2, 1, 3).reshape(Hkv * G, Lq, D)
        np.testing.assert_allclose(got, ref[:, n:, :], atol=1e-12)


def pin_attention_single_visible_key():
    """With no prefix, query token 0 sees only itself: o = v_q[0]."""
    rng = np.random.default_rng(8)
    D = 16
    kc = np.zeros((2, 0, D))
    q = rng.standard_normal((2, 3, 2, D))
    kq = rng.standard_normal((2, 3, D))
    vq = rng.standard_normal((2, 3, D))
    o = oracle.query_attention(kc, kc, q, kq, vq, 1e4)
    for g in range(2):
        np.testing.assert_allclose(o[:, 0, g], vq[:, 0], atol=1e-15)


def pin_attention_zero_query_is_mean():
    """A zero query gives equal weight to every visible row: o = mean(v)."""
    rng = np.random.default_rng(9)
    P, Lq, D = 11, 4, 8
    kc = rng.standard_normal((1, P, D))
    vc = rng.standard_normal((1, P, D))
    kq = rng.standard_normal((1, Lq, D))
    vq = rng.standard_normal((1, Lq, D))
    o = oracle.query_attention(kc, vc, np.zeros((1, Lq, 1, D)), kq, vq, 1e4)
    allv = np.concatenate([vc[0], vq[0]])
    for t in range(Lq):
        np.testing.assert_allclose(o[0, t, 0], allv[:P + t + 1].mean(0), atol=1e-14)


PINS = [pin_fig5_worked_example, pin_delta_formula_and_brute_force, pin_composite_positions,
        pin_rope_identity, pin_rope_vs_complex, pin_rope_closed_form,
        pin_rope_composition_and_norm, pin_rope_relative_position,
        pin_rope_interleaved, pin_interleaved_layout_is_a_relabelling,
        pin_assemble_is_rope_at_target, pin_unrotated_sources_take_rope_at_their_positions,
        pin_attention_single_chunk_is_causal_attention,
        pin_attention_single_visible_key, pin_attention_zero_query_is_mean]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_mod, pin):
    pin()
