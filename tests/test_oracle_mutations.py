"""Planted-mistake check for the oracle's pins (CPU only).

Each case copies the oracle's C source, plants one plausible mistake by a
text substitution, builds the copy in a temporary directory and requires at
least one of the named pins to fail against it. The committed oracle source
is never modified.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle.build import _HERE as ORACLE_DIR
from tests import test_oracle_pins as pins

SRC = open(os.path.join(ORACLE_DIR, "mxq_oracle.c")).read()

MUTATIONS = [
    ("ties away from zero", "double q = nearbyint(frac * 8.0);", "double q = round(frac * 8.0);",
     ["test_e4m3_ties_go_to_even"]),
    ("no saturation below 480", "if (a > 448.0) return sign | 0x7E;", "if (a > 480.0) return sign | 0x7E;",
     ["test_e4m3_known_points", "test_e4m3_encode_bruteforce_all_bf16"]),
    ("shared exponent off by one", "int s = (e - 1) - 8;", "int s = e - 8;",
     ["test_e8m0_exhaustive_bf16"]),
    ("no clamp of tiny exponents", "if (s < -127) s = -127;", "",
     ["test_e8m0_exhaustive_bf16"]),
    ("negative zero loses its sign", "uint8_t sign = signbit(v) ? 0x80 : 0;", "uint8_t sign = v < 0 ? 0x80 : 0;",
     ["test_e4m3_known_points"]),
    ("swizzle inner 4x4 transposed", "(r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4)",
     "(r % 32) * 16 + (c % 4) * 4 + ((r % 128) / 32)", ["test_swizzle_structure"]),
    ("colwise scale read transposed", "S_compact[(m / 32) * cc + k]", "S_compact[k * cr + m / 32]",
     ["test_dequant_matches_independent_decode"]),
    ("dgrad reads rowwise weight scales",
     "double b = deq_col(wq, ws, wc, K, (int64_t)e * N + n, k);",
     "double b = deq_row(wq, ws, wc, K, (int64_t)e * N + n, k);",
     ["test_gemms_match_blas_on_quantized_operands"]),
    ("wgrad drops the last row of each expert",
     "for (int64_t m = off; m < off + m_splits[e]; ++m) {\n            double a = deq_col",
     "for (int64_t m = off; m < off + m_splits[e] - 1; ++m) {\n            double a = deq_col",
     ["test_gemms_exact_on_small_integers"]),
    ("fprop ignores the bias", "if (bias) { double bb", "if (0) { double bb",
     ["test_gemms_match_blas_on_quantized_operands"]),
    ("dbias skips the last row", "for (int64_t m = off; m < off + m_splits[e]; ++m) acc += orc_bf16_value",
     "for (int64_t m = off + 1; m < off + m_splits[e]; ++m) acc += orc_bf16_value", ["test_grouped_dbias"]),
    ("swiglu gate and up swapped", "double g = orc_bf16_value(y[m * 2 * F + f]);\n            double u = orc_bf16_value(y[m * 2 * F + F + f]);\n            double sg = 1.0 / (1.0 + exp(-g));\n            h[",
     "double u = orc_bf16_value(y[m * 2 * F + f]);\n            double g = orc_bf16_value(y[m * 2 * F + F + f]);\n            double sg = 1.0 / (1.0 + exp(-g));\n            h[",
     ["test_swiglu_against_closed_forms"]),
    ("swiglu backward uses (1 + s) for (1 - s)", "d * u * sg * (1.0 + g * (1.0 - sg))",
     "d * u * sg * (1.0 + g * (1.0 + sg))", ["test_swiglu_against_closed_forms"]),
    ("swiglu backward du takes u for g", "dy[m * 2 * F + F + f] = orc_bf16_round(d * g * sg);",
     "dy[m * 2 * F + F + f] = orc_bf16_round(d * u * sg);", ["test_swiglu_against_closed_forms"]),
    ("scaled dbias drops the routing scale", "acc += (double)probs[m] * dy[m * N + n];", "acc += dy[m * N + n];",
     ["test_scaled_bias_grads_are_gradients_of_the_scaled_bias_term"]),
    ("routing-scale grad reads the next expert's bias", "acc += dy[m * N + n] * orc_bf16_value(bias[e * N + n]);",
     "acc += dy[m * N + n] * orc_bf16_value(bias[((e + 1) % E) * N + n]);",
     ["test_scaled_bias_grads_are_gradients_of_the_scaled_bias_term"]),
    ("routing-scale grad skips the last column",
     "for (int64_t n = 0; n < N; ++n) acc += dy[m * N + n] * orc_bf16_value(bias[e * N + n]);",
     "for (int64_t n = 0; n < N - 1; ++n) acc += dy[m * N + n] * orc_bf16_value(bias[e * N + n]);",
     ["test_scaled_bias_grads_are_gradients_of_the_scaled_bias_term"]),
    ("colwise blocks cross rows wrongly", "for (int t = 0; t < 32; ++t) v[t] = x[(32 * i + t) * K + k];",
     "for (int t = 0; t < 32; ++t) v[t] = x[(32 * i + t) * K + (k ^ 1)];",
     ["test_group_quantize_equals_blockwise_definition"]),
]


def _build_mutant(tmp_path, old, new):
    assert SRC.count(old) == 1, old
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    so = tmp_path / "libmutant.so"
    cmd = ["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-ffp-contract=off", "-fvisibility=hidden",
           str(src), "-o", str(so), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    oracle._declare(lib)
    return lib


@pytest.mark.parametrize("name,old,new,tests", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, tests):
    mutant = _build_mutant(tmp_path, old, new)
    saved = oracle._lib
    oracle._lib = mutant
    failed = []
    try:
        for t in tests:
            fn = getattr(pins, t)
            params = getattr(fn, "pytestmark", [])
            cases = [()]
            for mark in params:
                if mark.name == "parametrize":
                    argn, vals = mark.args[0], mark.args[1]
                    cases = [v if isinstance(v, tuple) else (v,) for v in vals]
            for case in cases:
                try:
                    fn(oracle, *case)
                except (AssertionError, ValueError):
                    failed.append(t)
                    break
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake: {name}"


def test_pins_catch_padding_to_32_rows(monkeypatch):
    """Planted mistake in the oracle's Python layer: experts padded to 32 rows instead of 128."""
    def wrong(m_splits):
        ms = np.asarray(m_splits, np.int64)
        mp = (ms + 31) // 32 * 32
        return np.concatenate([[0], np.cumsum(mp)]).astype(np.int64), mp

    monkeypatch.setattr(oracle, "padded_offsets", wrong)
    with pytest.raises((AssertionError, ValueError)):
        pins.test_padded_partial_colwise_block_by_brute_force(oracle)
