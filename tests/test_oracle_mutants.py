"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the oracle's C source (CPU only, in a temporary
directory), builds it, and runs the pin suite against that build through
ORACLE_LIB: the suite has to fail."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pagedkv_oracle.c")

MUTANTS = {
    "decode_gqa_mapping_modulo": ("h / group, num_kv_heads, page_size, head_dim,",
                                  "h % num_kv_heads, num_kv_heads, page_size, head_dim,"),
    "prefill_gqa_mapping_modulo": ("h / group, num_kv_heads, page_size, d_qk, d_vo,",
                                   "h % num_kv_heads, num_kv_heads, page_size, d_qk, d_vo,"),
    "sink_dropped_from_denominator": ("double den = has_sink ? exp(sink - m) : 0.0;",
                                      "double den = 0.0;"),
    "window_not_inclusive": ("lo = p - window_left;", "lo = p - window_left + 1;"),
    "decode_tokens_not_causal": ("int64_t p = L - Q + t;", "int64_t p = L - 1;"),
    "varlen_rows_from_request_start": ("t = (int)(row - cum_seq_lens_q[b]);", "t = 0;"),
    "varlen_uniform_length": ("Q = cum_seq_lens_q[b + 1] - cum_seq_lens_q[b];", "Q = q_len_per_req;"),
    "varlen_request_search_strict": ("if (cum_seq_lens_q[mid] <= row)", "if (cum_seq_lens_q[mid] < row)"),
    "prefill_top_left_causal": ("int64_t pos = kvb - qb + i;", "int64_t pos = i;"),
    "hnd_addressed_as_nhd": ("within = ((int64_t)head * page_size + slot) * head_dim + d;",
                             "within = ((int64_t)slot * num_kv_heads + head) * head_dim + d;"),
    "seq_len_ignores_last_page": (
        "seq_lens[b] = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;",
        "seq_lens[b] = pages > 0 ? pages * page_size : 0;"),
    "append_len_check_off_by_page": (
        "int len = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;",
        "int len = pages * page_size;"),
    "positions_from_zero": ("positions[i] = (int32_t)(seq_lens[b] - n + k);",
                            "positions[i] = (int32_t)k;"),
    "lse_missing_log_den": ("*lse = m + log(den);", "*lse = m;"),
    "bmm2_not_applied": ("o[d] = out_scale * o[d] / den;", "o[d] = o[d] / den;"),
    "logit_scale_dropped": ("s[jj] = scale * dot;", "s[jj] = dot;"),
    "fp16_exponent_bias": ("expo - 25);", "expo - 24);"),
    "merge_weights_unnormalised": ("double w = exp(lse_parts[i] - total);",
                                   "double w = exp(lse_parts[i] - m);"),
    "append_slot_shifted": ("int slot = p % page_size;", "int slot = (p + 1) % page_size;"),
    "e4m3_exponent_bias": ("v = ldexp((double)(8 + mant), expo - 10);",
                           "v = ldexp((double)(8 + mant), expo - 9);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)mant, -9);", "v = ldexp((double)mant, -10);"),
    "append_copies_half_the_bytes": ("(const char *)append_key + src * elem_bytes, elem_bytes);",
                                     "(const char *)append_key + src * elem_bytes, 1);"),
    "value_row_from_key_cache": ("o[d] += w * (v_mul * orc_elem(v_cache, off, kv_dtype));",
                                 "o[d] += w * (v_mul * orc_elem(k_cache, off, kv_dtype));"),
    "v_scale_not_applied": ("o[d] += w * (v_mul * orc_elem(v_cache, off, kv_dtype));",
                            "o[d] += w * orc_elem(v_cache, off, kv_dtype);"),
    "k_scale_used_for_q": ("dot += (q_mul * orc_elem(q, q_off + d, dtype)) * (k_mul * orc_elem(k_cache, off, kv_dtype));",
                           "dot += (k_mul * orc_elem(q, q_off + d, dtype)) * (k_mul * orc_elem(k_cache, off, kv_dtype));"),
    "decode_excludes_own_key": ("int64_t lo = 0, hi = p;", "int64_t lo = 0, hi = p - 1;"),
    "prefill_always_causal": ("int64_t hi = causal ? (pos < kvb - 1 ? pos : kvb - 1) : kvb - 1;",
                              "int64_t hi = pos < kvb - 1 ? pos : kvb - 1;"),
    "prefill_excludes_own_key": ("int64_t hi = causal ? (pos < kvb - 1 ? pos : kvb - 1) : kvb - 1;",
                                 "int64_t hi = causal ? (pos - 1 < kvb - 1 ? pos - 1 : kvb - 1) : kvb - 1;"),
    "bf16_decoded_as_fp16": ("return dtype == ORC_BF16 ? orc_from_bf16(h[i]) : orc_from_fp16(h[i]);",
                             "return orc_from_fp16(h[i]);"),
    "sink_scaled_by_logit_scale": ("sinks != NULL, sinks ? (double)sinks[h] : 0.0,",
                                   "sinks != NULL, sinks ? bmm1_scale * (double)sinks[h] : 0.0,"),
    "lse_in_base_two": ("*lse = m + log(den);", "*lse = m + log2(den);"),
    "prefill_query_read_as_cache_type": (
        "err |= orc_attend_row(q, r * d_qk, q_dtype, q_scale, k_scale, v_scale, k_cache, v_cache, kv_dtype,",
        "err |= orc_attend_row(q, r * d_qk, kv_dtype, q_scale, k_scale, v_scale, k_cache, v_cache, kv_dtype,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(lib),
                    str(mutant), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
