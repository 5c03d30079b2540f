"""Each pin set must catch a plausible slip in the oracle.

A mistake is planted in a copy of the oracle's C source (on the CPU, in a
temporary directory), the copy is compiled, and at least one pin must fail on
it.  This shows that the pins can tell a correct oracle from a nearly-correct
one: a dropped term, a wrong sign, a wrong index, a swapped operand.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "gqa_head_mapping": ("int j = h / group;\n            double *o = out",
                         "int j = h % num_kv_heads;\n            double *o = out"),
    "dropped_scale": ("s[p - p0] = scale * dot;", "s[p - p0] = dot;"),
    "block_offset_off_by_one": ("        int off = p % bs;\n        double dot",
                                "        int off = (p + 1) % bs;\n        double dot"),
    "scores_read_v": ("oracle_half_to_double(k_cache[cache_index(phys, j, off, d, Hkv, bs, D)]);\n        s[",
                      "oracle_half_to_double(k_cache[cache_index(phys, j, off, (d + 1) % D, Hkv, bs, D)]);\n        s["),
    "softmax_sign": ("double w = exp(s[p - p0] - m);", "double w = exp(m - s[p - p0]);"),
    "half_exponent_bias": ("expo - 25", "expo - 24"),
    "merge_drops_l": ("double w = l_part[row0 + p] * exp(m_part[row0 + p] - M);",
                      "double w = exp(m_part[row0 + p] - M);"),
    "append_offset": ("int off = (int)(slot % block_size);\n        for (int j = 0; j < num_kv_heads; ++j) {\n            for",
                      "int off = (int)(slot / block_size) % block_size;\n        for (int j = 0; j < num_kv_heads; ++j) {\n            for"),
    "append_kv_swapped": ("k_cache[dst] = k_new[src];\n                v_cache[dst] = v_new[src];",
                          "k_cache[dst] = k_new[src];\n                v_cache[dst] = k_new[src];"),
    "slot_uses_next_block": ("block_tables[(int64_t)b * max_blocks_per_seq + pos / block_size]",
                             "block_tables[(int64_t)b * max_blocks_per_seq + (pos + 1) / block_size]"),
    "kv_bytes_missing_factor": ("return 2 * batch * L * H * D * S * elem_bytes;",
                                "return batch * L * H * D * S * elem_bytes;"),
    "max_not_subtracted_in_l": ("        int off = p % bs;\n        l += w;\n", "        int off = p % bs;\n        l += w * w;\n"),
    "copy_blocks_drops_v": ("            v_cache[(int64_t)dst[i] * per_block + e] = v_cache[(int64_t)src[i] * per_block + e];\n",
                            ""),
    "quant_truncates": ("float r = rintf(", "float r = truncf("),
    "quant_step_128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "dequant_drops_scale": ("((double)k_codes[row * head_dim + d] * k_scale[row])",
                            "((double)k_codes[row * head_dim + d])"),
    "quant_append_head_zero": ("int64_t row = (blk * num_kv_heads + j) * block_size + off;",
                               "int64_t row = (blk * num_kv_heads) * block_size + off;"),
    "multi_misses_own_position": ("int visible = ctx - n + i + 1;", "int visible = ctx - n + i;"),
    "multi_row_offset": ("int64_t t = query_start[b] + i;", "int64_t t = query_start[b] + n - 1 - i;"),
    "swap_copy_wrong_index": ("dst_k[(int64_t)dst[i] * elems + e] = src_k[(int64_t)src[i] * elems + e];",
                              "dst_k[(int64_t)dst[i] * elems + e] = src_k[(int64_t)dst[i] * elems + e];"),
    "quant_kv_drops_v_scale": ("o[d] += w * ((double)v_codes[row * head_dim + d] * v_scale[row]);",
                               "o[d] += w * ((double)v_codes[row * head_dim + d]);"),
    "quant_kv_v_from_k": ("oracle_quantize_k_row(v_codes + row * head_dim, v_scale + row, v_new + src, head_dim);",
                          "oracle_quantize_k_row(v_codes + row * head_dim, v_scale + row, k_new + src, head_dim);"),
    "copy_blocks_one_head": ("int64_t per_block = (int64_t)num_kv_heads * block_size * head_dim;",
                             "int64_t per_block = (int64_t)block_size * head_dim;"),
    "e4m3_exponent_bias": ("v = ldexp((double)(8 + frac), expo - 10);", "v = ldexp((double)(8 + frac), expo - 11);"),
    "e4m3_subnormal_step": ("v = ldexp((double)frac, -9);", "v = ldexp((double)frac, -10);"),
    "e4m3_ties_to_odd": ("(above == below && ((lo + 1) & 1) == 0)", "(above == below && ((lo + 1) & 1) == 1)"),
    "e4m3_rounds_down": ("if (above < below || (above == below", "if (above < below - 1e300 || (above == below"),
    "e4m3_sign_dropped": ("return (uint8_t)(signbit(y) ? (best | 0x80) : best);", "return (uint8_t)best;"),
    "fp8_step_127": ("float s = amax / 448.0f;", "float s = amax / 127.0f;"),
    "fp8_v_from_k": ("oracle_quantize_fp8_row(v_codes + row * head_dim, v_scale + row, v_new + src, head_dim);",
                     "oracle_quantize_fp8_row(v_codes + row * head_dim, v_scale + row, k_new + src, head_dim);"),
    "fp8_keys_use_value_scale": ("(oracle_e4m3_to_double(k_codes[row * head_dim + d]) * k_scale[row])",
                                 "(oracle_e4m3_to_double(k_codes[row * head_dim + d]) * v_scale[row])"),
    "fp8_values_drop_scale": ("(oracle_e4m3_to_double(v_codes[row * head_dim + d]) * v_scale[row])",
                              "(oracle_e4m3_to_double(v_codes[row * head_dim + d]))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE, encoding="utf-8") as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new), encoding="utf-8")
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
