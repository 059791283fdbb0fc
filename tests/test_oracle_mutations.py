"""The oracle's pins have teeth: copies of the oracle with one planted mistake
each (a flipped sign, a wrong pairing or frequency, an off-by-one position, a
dropped mask, a transposed operand ...) are each caught by at least one pin.

Every mutant is built from ``oracle/kvr_oracle.c`` by one textual replacement
into a temporary library; the real oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "kvr_oracle.c")

MUTANTS = {
    "rotation_sign": ("out[r * D + i] = x1 * c - x2 * s;", "out[r * D + i] = x1 * c + x2 * s;"),
    "rotation_sign_2": ("out[r * D + i + h] = x1 * s + x2 * c;", "out[r * D + i + h] = -x1 * s + x2 * c;"),
    "interleaved_pairs": ("const int h = D / 2;", "const int h = 1;"),
    "frequency_exponent": ("pow(theta, -2.0 * (double)i / (double)D)", "pow(theta, -1.0 * (double)i / (double)D)"),
    "delta_is_target": ("delta[i] = target[i] - s.start;", "delta[i] = target[i];"),
    "inclusive_length": ("next += (int64_t)(s.end - s.start);", "next += (int64_t)(s.end - s.start + 1);"),
    "composite_from_zero": ("target[i] = composite ? s.start : next;", "target[i] = composite ? 0 : next;"),
    "mask_drops_self": ("const int64_t n_vis = P + t + 1;", "const int64_t n_vis = P + t;"),
    "no_causal_mask": ("const int64_t n_vis = P + t + 1;", "const int64_t n_vis = N;"),
    "query_key_position": ("const double sh = (double)(P + t);\n            rope_row(interleaved, D, kq",
                           "const double sh = (double)(P + t + 1);\n            rope_row(interleaved, D, kq"),
    "query_not_rotated": ("rope_row(interleaved, D, q + ((u * Lq + t) * G + g) * D, sh, theta, qr);",
                          "memcpy(qr, q + ((u * Lq + t) * G + g) * D, sizeof(double) * (size_t)D);"),
    "scale": ("scale = 1.0 / sqrt((double)D);", "scale = 1.0 / (double)D;"),
    "query_head_layout": ("q + ((u * Lq + t) * G + g) * D", "q + ((u * G + g) * Lq + t) * D"),
    "values_from_keys": ("acc += sc[j] * V[j * D + d];", "acc += sc[j] * K[j * D + d];"),
    "missing_normaliser": ("orow[d] = acc / z;", "orow[d] = acc;"),
    "interleaved_sign": ("yr[2 * i] = ev * cs - od * sn;", "yr[2 * i] = ev * cs + od * sn;"),
    "interleaved_frequency": ("shift[r] * inv_freq(theta, D, i);\n            const double cs",
                              "shift[r] * inv_freq(theta, D, 2 * i);\n            const double cs"),
    "interleaved_partner": ("const double ev = xr[2 * i], od = xr[2 * i + 1];",
                            "const double ev = xr[i], od = xr[i + D / 2];"),
    "interleaved_ignored": ("    if (interleaved)\n        kvo_rope_rows_interleaved", "    if (0)\n        kvo_rope_rows_interleaved"),
    "value_row_shift": ("memcpy(V + (P + t) * D, vq + (u * Lq + t) * D", "memcpy(V + (P + t) * D, vq + (u * Lq + (t + 1) % Lq) * D"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, source, tmp_path, name):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(src), "-lm"],
                   check=True, capture_output=True)
    caught = []
    with oracle.use_library(str(lib)):
        for pin in pins.PINS:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name!r}"
