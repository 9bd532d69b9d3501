"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/splitkv_oracle.c`` (a
dropped scale, a wrong KV-head map, a causal off-by-one, a wrong LSE, a sign
flip, a wrong page offset, an unnormalised merge, MLA values taken from the
wrong columns; in the key-set partial a causal off-by-one, a dropped scale, a
wrong LSE or KV-head map), builds it into a temporary library on the CPU, and
checks that at least one pin of ``test_oracle_attention`` /
``test_oracle_merge`` / ``test_oracle_interleaved`` fails.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle_attention as TA
from tests import test_oracle_fp8 as TF
from tests import test_oracle_interleaved as TI
from tests import test_oracle_merge as TM

SRC = os.path.join(os.path.dirname(oracle.__file__), "splitkv_oracle.c")

MUTANTS = {
    "drop_scale": ("scores[j - j0] = p->scale * dot;", "scores[j - j0] = dot;"),
    "kv_head_map": ("int kv_head = (p->kind == 0) ? h / group : 0;",
                    "int kv_head = (p->kind == 0) ? h % p->num_kv_heads : 0;"),
    "causal_off_by_one": ("int j1 = key_end < pos + 1 ? key_end : pos + 1;",
                          "int j1 = key_end < pos ? key_end : pos;"),
    "lse_without_max": ("double l = m + log(sum);", "double l = log(sum);"),
    "weight_sign": ("double w = exp(scores[j - j0] - l);", "double w = exp(l - scores[j - j0]);"),
    "page_offset": ("int off = j % p->page_size;", "int off = (j + 1) % p->page_size;"),
    "merge_unnormalised": ("double w = exp(lse_parts[r] - m) / denom;", "double w = exp(lse_parts[r] - m);"),
    "mla_value_columns": ("o[d] += w * (widen(vbase, p->kv_dtype, vo + d) * vscale);",
                          "o[d] += w * (widen(vbase, p->kv_dtype, vo + d + (p->kind ? p->head_dim_qk - p->head_dim_v : 0)) * vscale);"),
    # the FP8 KV cache: E4M3 decoding and per-tensor scales
    "e4m3_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_subnormal": ("ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)"),
    "k_scale_dropped": ("dot += widen(p->q, p->dtype, qrow + d) * (widen(p->k_cache, p->kv_dtype, ko + d) * p->k_scale);",
                        "dot += widen(p->q, p->dtype, qrow + d) * widen(p->k_cache, p->kv_dtype, ko + d);"),
    "v_scale_swapped": ("double vscale = (p->kind == 0) ? p->v_scale : p->k_scale;",
                        "double vscale = (p->kind == 0) ? p->k_scale : p->k_scale;"),
    # the key-set partial (round-robin shards)
    "keyset_causal": ("if (keys[t] >= 0 && keys[t] <= last_visible)", "if (keys[t] >= 0 && keys[t] < last_visible)"),
    "keyset_scale": ("scores[t] = qk * p->scale;", "scores[t] = qk;"),
    "keyset_lse": ("const double lse_keys = smax + log(denom);", "const double lse_keys = log(denom);"),
    "keyset_kv_head": ("const int kvh = (p->kind == 0) ? h / (p->num_q_heads / p->num_kv_heads) : 0;",
                       "const int kvh = (p->kind == 0) ? h % p->num_kv_heads : 0;"),
}

PINS = [
    lambda: TA.test_gqa_decode_matches_sdpa("f32"),
    TA.test_mla_matches_sdpa_with_shared_latent,
    TA.test_causal_prefill_matches_sdpa_and_chunk_rows_match_prefill_rows,
    TA.test_closed_forms,
    TA.test_partial_key_ranges_and_empty_subset,
    lambda: TM.test_merge_of_any_partition_equals_unsplit(3),
    TM.test_merge_hand_computed_two_states,
    TI.test_range_key_set_equals_range_partial,
    TI.test_scattered_key_set_matches_torch_attention,
    lambda: TI.test_merge_of_round_robin_partials_equals_unsplit(3),
    TF.test_e4m3_decoder_matches_torch_on_every_code,
    TF.test_fp8_attention_matches_sdpa_on_dequantized_cache,
    TF.test_fp8_scales_closed_forms,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mut = tmp_path / f"mut_{name}.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / f"libmut_{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(mut), "-lm"],
                   check=True)
    failures = 0
    with oracle.use_library(str(lib)):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


def test_unmutated_source_passes_all_pins():
    for pin in PINS:
        pin()
