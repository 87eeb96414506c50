"""Plant plausible mistakes in (a copy of) the oracle and check that the pins catch each.

Every mutant is the oracle's C source with one textual edit, compiled on the CPU into a
temporary library and swapped in for the duration of the test. A mutant that passes
every pin would mean the pins do not constrain that part of the oracle.
"""
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_prep_pins as prep_pins
import test_oracle_quant_pins as qpins

MUTANTS = [
    ("GQA head mapping h % kvh instead of h / G", "h / G", "h % kvh"),
    ("causal limit one short", "(int64_t)past[b] + j, rows", "(int64_t)past[b] + j - 1, rows"),
    ("scale dropped from the scores", "scores[t] = scale * dot;", "scores[t] = dot;"),
    ("default scale 1/head_size", "1.0 / sqrt((double)hs)", "1.0 / (double)hs"),
    ("wrong sign in the max shift", "double w = exp(scores[t] - m);", "double w = exp(scores[t] + m);"),
    ("lse in base 2", "*lse = m + log(den);", "*lse = m + log2(den);"),
    ("offsets reversed inside a page", "rows[t] = blk * bs + t % bs;", "rows[t] = blk * bs + (bs - 1 - t % bs);"),
    ("slot ignores past_seqlens", "int64_t p = (int64_t)past[b] + (i - cum[b]);", "int64_t p = (i - cum[b]);"),
    ("packed K taken from the wrong head offset", "query + i * qw + (int64_t)nh * hs : key",
     "query + i * qw + (int64_t)(nh - 1) * hs : key"),
    ("-1 slots not skipped", "if (slot == -1) continue;", ""),
    ("rounding truncates", "if (rem > half || (rem == half && (kept & 1))) kept += 1;", ""),
    ("PV unweighted", "out[d] += w * kv_value(kv_v, rows[t], g, kvh, hs, d);",
     "out[d] += kv_value(kv_v, rows[t], g, kvh, hs, d);"),
    ("normalisation dropped", "for (int d = 0; d < hs; ++d) out[d] /= den;", ""),
    ("fp16 exponent bias off by one", "ldexp((double)(m | 0x400), e - 25)", "ldexp((double)(m | 0x400), e - 24)"),
    ("bf16 decoded as the low half", "int sign = (h >> 15) & 1, e = (h >> 7) & 0xFF, m = h & 0x7F;",
     "int sign = (h >> 15) & 1, e = (h >> 6) & 0xFF, m = h & 0x3F;"),
    ("V read from the K cache", "vv = {0, value_cache, tab, NULL, NULL};\n  rc = attention_all(",
     "vv = {0, key_cache, tab, NULL, NULL};\n  rc = attention_all("),
    ("rotation sign flipped", "y[u] = a * ca[u] - b * sa[u];", "y[u] = a * ca[u] + b * sa[u];"),
    ("rotation pairs neighbours", "const double a = y[u], b = y[u + d / 2];\n    y[u] = a * ca[u] - b * sa[u];\n    y[u + d / 2] = b * ca[u] + a * sa[u];",
     "if (2 * u + 1 >= d) continue;\n    const double a = y[2 * u], b = y[2 * u + 1];\n    y[2 * u] = a * ca[u] - b * sa[u];\n    y[2 * u + 1] = b * ca[u] + a * sa[u];"),
    ("rotary angle in fp64", "const float ang = (float)pos * freq;", "const double ang = (double)pos * pow(base, -2.0 * u / rotary_dim);"),
    ("frequency exponent without the factor 2", "(float)pow(base, -2.0 * u / rotary_dim)", "(float)pow(base, -1.0 * u / rotary_dim)"),
    ("RMSNorm without the square root", "r = 1.0 / sqrt(ss / hs + eps);", "r = 1.0 / (ss / hs + eps);"),
    ("RMSNorm eps dropped", "r = 1.0 / sqrt(ss / hs + eps);", "r = 1.0 / sqrt(ss / hs);"),
    ("position without past_seqlens", "const int64_t pos = (int64_t)past[lo] + (i - cum[lo]);",
     "const int64_t pos = (int64_t)(i - cum[lo]);"),
    ("gate sign flipped", "gated[i] = out[i] / (1.0 + exp(-tab[gate[i]]));", "gated[i] = out[i] / (1.0 + exp(tab[gate[i]]));"),
    ("gate without the one", "gated[i] = out[i] / (1.0 + exp(-tab[gate[i]]));", "gated[i] = out[i] / exp(-tab[gate[i]]);"),
    ("quantization truncates", "float r = rintf(x / s);", "float r = truncf(x / s);"),
    ("quantization multiplies by the scale", "float r = rintf(x / s);", "float r = rintf(x * s);"),
    ("quantization clamps one past Q", "r = fmaxf(r, (float)-qmax);", "r = fmaxf(r, (float)(-qmax - 1));"),
    ("quantization with KV head 0's scales", "scale[(int64_t)g * hs + d], qmax)", "scale[d], qmax)"),
    ("INT4 written high nibble first", "((d & 1) ? 4 : 0)", "((d & 1) ? 0 : 4)"),
    ("INT4 read high nibble first", "int nib = (d & 1) ? row[d / 2] >> 4 : row[d / 2] & 0x0F;",
     "int nib = (d & 1) ? row[d / 2] & 0x0F : row[d / 2] >> 4;"),
    ("INT4 read without the sign", "return nib >= 8 ? nib - 16 : nib;", "return nib;"),
    ("INT8 read unsigned", "(double)(int8_t)v->codes[", "(double)v->codes["),
    ("dequantized with KV head 0's scales", "const double s = (double)v->scale[(int64_t)g * hs + d];",
     "const double s = (double)v->scale[d];"),
    ("V codes written into the K cache", "memcpy(value_cache + slots[i] * row_bytes, v_codes",
     "memcpy(value_cache + slots[i] * row_bytes, k_codes"),
]

# a fast battery of pins (each raises on failure)
BATTERY = [
    lambda: pins.test_prefill_from_empty_matches_sdpa_causal("fp16", 4, 2, 64, 16),
    lambda: pins.test_prefill_from_empty_matches_sdpa_causal("bf16", 6, 2, 32, 8),
    lambda: pins.test_decode_matches_sdpa_without_mask("bf16"),
    lambda: pins.test_chunked_prefill_matches_sdpa_bottom_right_mask("fp16"),
    lambda: pins.test_single_token_no_past_returns_its_own_v("fp16"),
    lambda: pins.test_single_token_no_past_returns_its_own_v("bf16"),
    lambda: pins.test_two_keys_closed_forms("fp16"),
    lambda: pins.test_constant_v_returns_v("bf16"),
    lambda: pins.test_slot_golden_table(),
    lambda: pins.test_minus_one_slots_leave_cache_untouched_and_reads_use_cache(),
    lambda: pins.test_packed_qkv_equals_separate(),
    lambda: pins.test_scale_zero_means_inverse_sqrt_head_size(),
    lambda: prep_pins.test_position_zero_is_identity(),
    lambda: prep_pins.test_rotation_keeps_every_pair_length(32),
    lambda: prep_pins.test_scores_depend_on_the_position_difference_only(),
    lambda: prep_pins.test_rms_norm_with_unit_and_general_weights(),
    lambda: prep_pins.test_single_component_rotates_into_its_half_partner(1),
    lambda: prep_pins.test_single_component_rotates_into_its_half_partner(7),
    lambda: prep_pins.test_gate_closed_forms("fp16"),
    lambda: prep_pins.test_gate_symmetry(),
    lambda: qpins.test_exact_multiples_give_their_integer("int8", "fp16"),
    lambda: qpins.test_exact_multiples_give_their_integer("int4", "bf16"),
    lambda: qpins.test_halfway_values_round_to_even("int8"),
    lambda: qpins.test_saturation_zero_and_nan("int8"),
    lambda: qpins.test_saturation_zero_and_nan("int4"),
    lambda: qpins.test_quantization_matches_numpy_float32("int8", "bf16"),
    lambda: qpins.test_quantization_matches_numpy_float32("int4", "fp16"),
    lambda: qpins.test_int4_nibble_order_by_hand(),
    lambda: qpins.test_int8_bytes_by_hand(),
    lambda: qpins.test_attention_equals_the_16bit_operator_on_exact_values("int8", "fp16"),
    lambda: qpins.test_attention_equals_the_16bit_operator_on_exact_values("int4", "bf16"),
    lambda: qpins.test_one_key_returns_its_dequantized_value("int8"),
    lambda: qpins.test_one_key_returns_its_dequantized_value("int4"),
    lambda: qpins.test_scores_use_the_k_scale_of_each_channel("int4"),
    lambda: qpins.test_cache_write_places_code_rows_and_skips_dropped_slots("int8"),
]


def _compile_mutant(tmp_path, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    return str(so)


def test_battery_passes_on_the_real_oracle():
    for pin in BATTERY:
        pin()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_each_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name, old, new):
    lib = oracle._bind(_compile_mutant(tmp_path, old, new))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    with np.errstate(all="ignore"):
        for k, pin in enumerate(BATTERY):
            try:
                pin()
            except (AssertionError, oracle.OracleError, ValueError, FloatingPointError):
                caught.append(k)
    assert caught, f"no pin caught the mutant: {name}"
