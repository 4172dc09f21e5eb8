"""The oracle's pins must catch plausible slips.

Each case plants one mistake in a copy of oracle.c (compiled on the CPU into a
temporary directory), runs the pin tests against the mutant and requires at
least one of them to fail.  The mutations never move a memory access out of
bounds.
"""
import functools
import os
import subprocess
import types

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTATIONS = {
    "causal_bound_drops_self": ("const int last = pb->causal ? P + i : Lk - 1;",
                                "const int last = pb->causal ? (i > 0 ? P + i - 1 : P + i) : Lk - 1;"),
    "gqa_interleaved_heads": ("const int kvh = h / (pb->n_heads / pb->n_kv_heads);",
                              "const int kvh = h % pb->n_kv_heads;"),
    "scale_dropped": ("s[j] = pb->scale * dot;", "s[j] = dot;"),
    "scale_divides": ("s[j] = pb->scale * dot;", "s[j] = dot / pb->scale;"),
    "first_key_dropped_from_sum": ("for (int j = first; j <= last; ++j)\n        Z += exp(s[j] - m);",
                                   "for (int j = first + (last > first); j <= last; ++j)\n        Z += exp(s[j] - m);"),
    "window_one_key_short": ("P + i - pb->window + 1 > 0) ? P + i - pb->window + 1 : 0;",
                             "P + i - pb->window + 2 > 0) ? P + i - pb->window + 2 : 0;"),
    "window_ignores_prefix": ("P + i - pb->window + 1 > 0) ? P + i - pb->window + 1 : 0;",
                              "i - pb->window + 1 > 0) ? P + i - pb->window + 1 : P;"),
    "value_read_from_keys": ("load_key(pb, 1, b, kvh, j, 0, kv);", "load_key(pb, 0, b, kvh, j, 0, kv);"),
    "lse_without_max": ("pb->lse[t * pb->n_heads + h] = m + log(Z);",
                        "pb->lse[t * pb->n_heads + h] = log(Z);"),
    "cache_written_at_zero": ("const size_t row = cache_row(&pb, b, kvh, P + i);",
                              "const size_t row = cache_row(&pb, b, kvh, i);"),
    "prefix_keys_shifted": ("const size_t row = cache_row(pb, b, kvh, j);",
                            "const size_t row = cache_row(pb, b, kvh, j > 0 ? j - 1 : 0);"),
    # paged cache (every mutant stays inside the pool: the pin tables fill every entry)
    "paged_row_off_by_one": ("(size_t)(pos % pb->block_size);", "(size_t)((pos + 1) % pb->block_size);"),
    "paged_pool_heads_outer": ("((size_t)blk * pb->n_kv_heads + kvh) * pb->block_size",
                               "((size_t)kvh * pb->num_blocks + blk) * pb->block_size"),
    "paged_table_of_first_seq": ("pb->block_table[(size_t)b * pb->max_blocks + pos / pb->block_size]",
                                 "pb->block_table[pos / pb->block_size]"),
    # rotary embedding
    "rope_interleaved_pairs": ("""        const double a = x[i], b = x[i + half];
        x[i] = a * c[i] - b * sn[i];
        x[i + half] = b * c[i] + a * sn[i];""", """        const double a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = a * c[i] - b * sn[i];
        x[2 * i + 1] = b * c[i] + a * sn[i];"""),
    "rope_rotates_backwards": ("""        x[i] = a * c[i] - b * sn[i];
        x[i + half] = b * c[i] + a * sn[i];""", """        x[i] = a * c[i] + b * sn[i];
        x[i + half] = b * c[i] - a * sn[i];"""),
    "rope_frequency_exponent_halved": ("powf((float)rope_theta, (float)(2 * i) / (float)head_dim)",
                                       "powf((float)rope_theta, (float)(i) / (float)head_dim)"),
    "rope_query_position_without_prefix": ("rope_rotate_bf16(pb, P + i, qv);", "rope_rotate_bf16(pb, i, qv);"),
    "rope_key_position_without_prefix": ("rope_rotate_bf16(pb, j, dst);", "rope_rotate_bf16(pb, j - pb->off[b], dst);"),
    "rope_cache_keeps_unrotated_key": ("if (c == 0 && pb.rope_cos) {", "if (0 && pb.rope_cos) {"),
    # int8 cache
    "quant_scale_over_128": ("const float sc = amax / 127.0f;", "const float sc = amax / 128.0f;"),
    "quant_truncates": ("qv = rintf((float)bf16_to_double(x[e]) / sc);", "qv = truncf((float)bf16_to_double(x[e]) / sc);"),
    "quant_dequant_drops_scale": ("dst[e] = (double)codes[e] * sc;", "dst[e] = (double)codes[e];"),
    "quant_scale_from_first_element": ("if (a > amax)\n                            amax = a;",
                                       "if (e == 0)\n                            amax = a;"),
}

PIN_TESTS = [
    pins.test_packed_equals_each_sequence_alone,
    pins.test_length_one_returns_v_and_score,
    pins.test_two_keys_is_a_logistic_blend,
    pins.test_causal_rows_sum_to_one,
    pins.test_equal_keys_give_prefix_mean,
    pins.test_gqa_contiguous_head_groups,
    pins.test_causality,
    pins.test_cache_write_closed_form,
    pins.test_toy_shapes_and_decode_append,
    functools.partial(pins.test_matches_torch_sdpa_float64, case="r3", causal=True),
    pins.test_window_closed_forms,
    functools.partial(pins.test_window_matches_torch_sdpa_float64, window=37),
    functools.partial(pins.test_paged_equals_contiguous, bs=16, seed=1),
    functools.partial(pins.test_paged_equals_contiguous, bs=5, seed=2),
    pins.test_rope_position_zero_is_identity,
    functools.partial(pins.test_rope_closed_form_rotations, m=7),
    pins.test_rope_relative_position_invariance,
    pins.test_rope_chunked_equals_one_shot,
    pins.test_rope_matches_complex_rotation_and_sdpa,
    pins.test_quant_codes_closed_form,
    pins.test_quant_rounding_bound_and_extremes,
    pins.test_quant_prefix_read_matches_sdpa_on_dequantised_cache,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    cmd = oracle.build_command()
    cmd[cmd.index(oracle._SRC)] = str(mutant_src)
    cmd[cmd.index(oracle._LIB_PATH)] = str(so)
    subprocess.check_call(cmd)
    lib = oracle.load_library(str(so))
    mutant = types.SimpleNamespace(prefill_attention=functools.partial(oracle.prefill_attention, lib=lib))
    failures = 0
    for t in PIN_TESTS:
        try:
            t(mutant)
        except Exception:  # an assertion, a rejected call or an overflow all count
            failures += 1
    assert failures >= 1, f"no pin caught mutation {name}"
