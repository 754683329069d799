"""Planted mistakes: each mutant of the oracle's C source must fail some pin.

Every mutant is compiled on the CPU into a temporary library, swapped in for
the real oracle for the duration of one check, and the pins of
test_oracle_pins.py are run against it.  A mutant that passes every pin would
mean the pins cannot see that kind of mistake.
"""
import ctypes
import os
import subprocess

import pytest
import torch

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sdpa_oracle.c")

MUTANTS = {
    "causal_edge_off_by_one": ("if (causal && j > p) return 0;", "if (causal && j >= p) return 0;"),
    "window_edge_off_by_one": ("if (window > 0 && p - j >= window) return 0;",
                               "if (window > 0 && p - j > window) return 0;"),
    "top_left_alignment": ("const int64_t p = (int64_t)Lk - Lq + i;", "const int64_t p = i;"),
    "gqa_modulo_head_map": ("  int g = h / G;\n  const int64_t qoff", "  int g = h % Hkv;\n  const int64_t qoff"),
    "half_contraction": ("for (int d = 0; d < Dqk; ++d) acc +=", "for (int d = 0; d < Dqk / 2; ++d) acc +="),
    "fp16_exponent_bias": ("mag = ldexp((double)(1024 + m), e - 25);", "mag = ldexp((double)(1024 + m), e - 24);"),
    "bf16_truncated_mantissa": ("uint32_t bits = (uint32_t)b << 16;", "uint32_t bits = (uint32_t)(b & 0xFFF0) << 16;"),
    "softmax_not_normalised": ("for (int64_t j = 0; j < Lk; ++j) P[j] /= den;", "(void)den;"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "bias_subtracted": ("if (brow) s[j] += elem(", "if (brow) s[j] -= elem("),
    "bias_scaled": ("if (brow) s[j] += elem(brow, j, dtype);",
                    "if (brow) s[j] += scale * elem(brow, j, dtype);"),
    "bias_head_stride_ignored": ("bias + b * sb + h * sh + i * sq", "bias + b * sb + i * sq"),
}

PIN_CHECKS = [
    lambda: pins.test_matches_torch_sdpa_float64(pins.CASES[2], torch.float16),
    lambda: pins.test_matches_torch_sdpa_float64(pins.CASES[3], torch.bfloat16),
    lambda: pins.test_matches_torch_sdpa_float64(pins.CASES[1], torch.float16),
    lambda: pins.test_window_one_returns_own_value(5, 40),
    lambda: pins.test_zero_query_gives_mean_of_visible_values(6),
    lambda: pins.test_gqa_equals_mha_with_repeated_kv_heads(),
    lambda: pins.test_input_widening_is_exact(torch.float16),
    lambda: pins.test_input_widening_is_exact(torch.bfloat16),
    lambda: pins.test_probability_rows_sum_to_one(True, 5),
    lambda: pins.test_two_key_worked_example(),
    lambda: pins.test_log_weight_bias_with_zero_query_gives_weighted_mean(),
    lambda: pins.test_bias_matches_torch_sdpa_float_mask((2, 4, 9), torch.float16),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", str(so),
                    str(c), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    real = oracle._load()
    so = _build_mutant(tmp_path, name, *MUTANTS[name])
    lib = ctypes.CDLL(so)
    for fn in ("oracle_sdpa", "oracle_sdpa_bias", "oracle_row_scores", "oracle_row_probs",
               "oracle_max_threads"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failures = 0
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught mutant {name}"
