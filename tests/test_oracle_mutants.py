"""The oracle's pins must catch plausible mistakes.  Each case copies the
oracle source, plants one mistake (on the CPU, in a temporary build), and
runs the pin suite against that build: the suite has to fail."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "interleaved_gqa_heads": (
        "for (int32_t h = g * group; h < (g + 1) * group; ++h)",
        "for (int32_t h = g; h < Hq; h += Hkv)"),
    "causal_excludes_self": ("for (int32_t j = 0; j <= p; ++j) {\n                double dot",
                             "for (int32_t j = 0; j < p; ++j) {\n                double dot"),
    "slot_uses_block_not_offset": ("phys * block_size + pos % block_size",
                                   "phys * block_size + pos / block_size"),
    "position_ignores_computed": ("int32_t pos = c + i;", "int32_t pos = i;"),
    "logits_first_token": ("logits_indices[r] = query_start_loc[r + 1] - 1;",
                           "logits_indices[r] = query_start_loc[r];"),
    "scale_dropped": ("w[j] = jb->scale * dot;", "w[j] = dot;"),
    "softmax_sign_flipped": ("w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);"),
    "cache_head_major_layout": (
        "int64_t dst = (slot * num_kv_heads + h) * head_dim + d;",
        "int64_t dst = ((int64_t)h * num_slots + slot) * head_dim + d;"),
    "top_left_causal": ("return jb->seq_lens[r] - q_len + (t - jb->query_start_loc[r]);",
                        "return (t - jb->query_start_loc[r]);"),
    "bf16_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "fp16_bias": ("expo - 25", "expo - 24"),
    "qsl_tail_zero": ("query_start_loc[i] = num_tokens;", "query_start_loc[i] = 0;"),
    "pv_reads_keys": ("acc += w[j] * vc[", "acc += w[j] * kc["),
    "seq_len_without_new_tokens": ("seq_lens[r] = c + n;", "seq_lens[r] = c;"),
    "token_index_row_stride": ("(int64_t)req_indices[t] * max_model_len;",
                               "(int64_t)req_indices[t] * max_num_reqs;"),
    "discard_when_caught_up": ("optimistic_seq_len < (int64_t)request_num_tokens[r];",
                               "optimistic_seq_len <= (int64_t)request_num_tokens[r];"),
    "discard_ignores_scheduled": (
        "(int64_t)num_computed_tokens[r] + (int64_t)num_scheduled_tokens[r];",
        "(int64_t)num_computed_tokens[r];"),
    "spec_rows_from_slice_start": ("logits_indices[row++] = last - d + k;",
                                   "logits_indices[row++] = query_start_loc[r] + k;"),
    "spec_drafts_ignored": ("int32_t d = num_draft_tokens ? num_draft_tokens[r] : 0;",
                            "int32_t d = 0;"),
    "copy_k_into_v": (
        "value_cache[(int64_t)d * block_bytes + b] = value_cache[(int64_t)s * block_bytes + b];",
        "value_cache[(int64_t)d * block_bytes + b] = key_cache[(int64_t)s * block_bytes + b];"),
    "copy_half_block": ("        for (int64_t b = 0; b < block_bytes; ++b) {\n            key_cache[(int64_t)d",
                        "        for (int64_t b = 0; b < block_bytes / 2; ++b) {\n            key_cache[(int64_t)d"),
    "zero_k_only": ("            value_cache[(int64_t)blk * block_bytes + b] = 0;\n", ""),
    "e4m3_bias": ("ldexp((double)(8 + mant), expo - 10)", "ldexp((double)(8 + mant), expo - 11)"),
    "e4m3_subnormal_scale": ("ldexp((double)mant, -9);", "ldexp((double)mant, -10);"),
    "e4m3_no_saturation": ("if (a >= 448.0)\n        return sign | 0x7e;",
                           "if (a >= 1e300)\n        return sign | 0x7e;"),
    "e4m3_ties_away": ("double steps = nearbyint(ldexp(a, 3 - e));",
                       "double steps = round(ldexp(a, 3 - e));"),
    "fp8_write_multiplies": ("float kq = (float)elem(key[src], src_dtype) / k_scale;",
                             "float kq = (float)elem(key[src], src_dtype) * k_scale;"),
    "fp8_v_scale_ignored": ("cache_elem(jb->value_cache, a, jb->cache_dtype) * jb->v_scale;",
                            "cache_elem(jb->value_cache, a, jb->cache_dtype);"),
    "gather_wrong_offset": ("int64_t slot = (int64_t)phys * jb->block_size + j % jb->block_size;",
                            "int64_t slot = (int64_t)phys * jb->block_size + j / jb->block_size;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "pa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libpa_oracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, PA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
