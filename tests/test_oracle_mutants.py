"""The oracle's pins catch plausible mistakes.

Each mutant is a copy of ``oracle/pa_oracle.c`` with one deliberate,
plausible error (a dropped term, a wrong sign, a wrong index, a transposed
operand).  It is compiled with gcc into a temporary library and the whole
pin suite runs against it in a child process; the test passes when at least
one pin fails (or the mutant crashes).  Mistakes are planted only in the
oracle, on the CPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

# (name, exact text in the source, replacement, occurrence index)
MUTANTS = [
    ("slot_offset_uses_logical",
     "return physical_block * block_size + offset;",
     "return physical_block * block_size + logical_block;", 0),
    ("slot_offset_divides",
     "    int64_t offset = position % block_size;\n    int64_t physical_block = block_table_row",
     "    int64_t offset = position / block_size;\n    int64_t physical_block = block_table_row", 0),
    ("slot_table_indexed_by_offset",
     "int64_t physical_block = block_table_row[logical_block];",
     "int64_t physical_block = block_table_row[offset];", 0),
    ("cache_writes_key_into_value",
     "value_cache[dst_i] = value[src_i];",
     "value_cache[dst_i] = key[src_i];", 0),
    ("cache_head_major_layout",
     "int64_t dst = (block * block_size + offset) * row_elems;",
     "int64_t dst = (offset * block_size + block) * row_elems;", 0),
    ("copy_blocks_only_keys",
     "            value_cache[dst * block_elems + i] = value_cache[src * block_elems + i];\n",
     "", 0),
    ("copy_blocks_reversed",
     "key_cache[dst * block_elems + i] = key_cache[src * block_elems + i];",
     "key_cache[src * block_elems + i] = key_cache[dst * block_elems + i];", 0),
    ("attention_drops_scale",
     "scores[p - p0] = scale * dot;",
     "scores[p - p0] = dot;", 0),
    ("attention_softmax_sign",
     "scores[j] = exp(scores[j] - m);",
     "scores[j] = exp(m - scores[j]);", 0),
    ("attention_no_normalise",
     "        out[i] /= l;",
     "        out[i] /= 1.0;", 0),
    ("attention_gqa_modulo",
     "                         h / group, num_kv_heads, head_dim, block_size, scale,",
     "                         h % num_kv_heads, num_kv_heads, head_dim, block_size, scale,", 0),
    ("attention_context_off_by_one",
     "row, 0, ctx,",
     "row, 0, ctx - 1,", 0),
    ("attention_head_major_cache",
     "return ((physical_block * block_size + offset) * num_kv_heads + kv_head) *",
     "return ((physical_block * num_kv_heads + kv_head) * block_size + offset) *", 0),
    ("attention_value_uses_key_pool",
     "out[i] += scores[j] * decode(value_cache[v + i], dtype);",
     "out[i] += scores[j] * decode(key_cache[v + i], dtype);", 0),
    ("attention_query_row_of_kv_head",
     "const uint16_t *q_row = query + ((int64_t)s * num_heads + h) * head_dim;\n            double m, l;",
     "const uint16_t *q_row = query + ((int64_t)s * num_heads + h / group) * head_dim;\n            double m, l;", 0),
    ("merge_drops_l",
     "double w = part_l[base + j] * exp(part_m[base + j] - big_m);",
     "double w = exp(part_m[base + j] - big_m);", 0),
    ("merge_no_stabiliser",
     "double w = part_l[base + j] * exp(part_m[base + j] - big_m);",
     "double w = part_l[base + j] * exp(part_m[base + j]);", 0),
    ("partition_end_unclipped",
     "                if (p1 > ctx)\n                    p1 = ctx;\n",
     "", 0),
    ("partition_count_floor",
     "return (int)((context_len + partition_size - 1) / partition_size);",
     "return (int)(context_len / partition_size);", 0),
    ("f16_subnormal_scale",
     "mag = ldexp((double)frac, -24);",
     "mag = ldexp((double)frac, -25);", 0),
    ("f16_exponent_bias",
     "mag = ldexp((double)(1024 + frac), expo - 25);",
     "mag = ldexp((double)(1024 + frac), expo - 24);", 0),
    ("bf16_shift",
     "uint32_t w = ((uint32_t)bits) << 16;",
     "uint32_t w = ((uint32_t)bits) << 15;", 0),
    ("empty_context_not_zero",
     "            if (ctx <= 0) {\n                for (int i = 0; i < head_dim; ++i)\n                    o[i] = 0.0;",
     "            if (ctx <= 0) {\n                for (int i = 0; i < head_dim; ++i)\n                    o[i] = 1.0;", 0),
    ("e4m3_decode_bias",
     "mag = ldexp((double)(8 + frac), expo - 10);",
     "mag = ldexp((double)(8 + frac), expo - 11);", 0),
    ("e4m3_encode_truncates",
     "double q = nearbyint(a / spacing);",
     "double q = floor(a / spacing);", 0),
    ("e4m3_saturates_low",
     "        return sign | 0x7e; /* 448 = 1.75 * 2^8, the largest finite value */",
     "        return sign | 0x7d; /* 448 = 1.75 * 2^8, the largest finite value */", 0),
    ("fp8_attention_drops_k_scale",
     "dot += decode(q_row[i], dtype) * (decode_e4m3(key_cache[k + i]) * k_scale);",
     "dot += decode(q_row[i], dtype) * decode_e4m3(key_cache[k + i]);", 0),
    ("fp8_attention_value_scale_is_k_scale",
     "o[i] += scores[p] * (decode_e4m3(value_cache[v + i]) * v_scale);",
     "o[i] += scores[p] * (decode_e4m3(value_cache[v + i]) * k_scale);", 0),
    ("prefill_excludes_own_token",
     "                             0, pos + 1, h / group, num_kv_heads, head_dim, block_size,",
     "                             0, pos, h / group, num_kv_heads, head_dim, block_size,", 0),
    ("prefill_positions_from_chunk_start",
     "int64_t pos = ctx - q_len + i;",
     "int64_t pos = i;", 0),
    ("prefill_query_row_unshifted",
     "int64_t r = (q0 + i) * num_heads + h;",
     "int64_t r = i * num_heads + h;", 0),
    ("fp8_cache_swaps_scales",
     "                             dtype, k_inv_scale);",
     "                             dtype, v_inv_scale);", 0),
    ("fp8_prefill_excludes_own_token",
     "                int64_t n = pos + 1;\n                double *scores = (double *)malloc(sizeof(double) * (size_t)n);",
     "                int64_t n = pos;\n                double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));", 0),
    ("fp8_prefill_value_scale_is_k_scale",
     "o[c] += scores[p] * (decode_e4m3(value_cache[v + c]) * v_scale);",
     "o[c] += scores[p] * (decode_e4m3(value_cache[v + c]) * k_scale);", 0),
    ("fp8_prefill_positions_from_chunk_start",
     "            int64_t pos = ctx - q_len + i;\n            for (int h = 0; h < num_heads; ++h) {\n                int64_t r = (q0 + i) * num_heads + h;\n                double *o = out + r * head_dim;\n                for (int k = 0; k < head_dim; ++k)",
     "            int64_t pos = i;\n            for (int h = 0; h < num_heads; ++h) {\n                int64_t r = (q0 + i) * num_heads + h;\n                double *o = out + r * head_dim;\n                for (int k = 0; k < head_dim; ++k)", 0),
    ("copy_blocks_u8_swapped",
     "        memcpy(key_cache + dst * block_elems, key_cache + src * block_elems,",
     "        memcpy(key_cache + src * block_elems, key_cache + dst * block_elems,", 0),
    ("copy_blocks_u8_half_block",
     "        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems,\n"
     "               (size_t)block_elems);",
     "        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems,\n"
     "               (size_t)block_elems / 2);", 0),
    ("copy_blocks_u8_only_keys",
     "        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems,\n"
     "               (size_t)block_elems);\n",
     "", 0),
    ("copy_blocks_u8_block_without_heads",
     "    int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;\n"
     "    for (int p = 0; p < num_pairs; ++p) {\n        int64_t src = block_mapping[2 * p];\n"
     "        int64_t dst = block_mapping[2 * p + 1];\n        memcpy(",
     "    int64_t block_elems = (int64_t)block_size * head_dim;\n"
     "    for (int p = 0; p < num_pairs; ++p) {\n        int64_t src = block_mapping[2 * p];\n"
     "        int64_t dst = block_mapping[2 * p + 1];\n        memcpy(", 0),
]

RUNNER = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
lib = oracle.load({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(lib)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED_PINS", ",".join(failed))
"""


def _mutate(text, old, new, occurrence):
    idx = -1
    for _ in range(occurrence + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutation anchor not found: {old!r}"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    csrc = tmp_path / f"{name}.c"
    csrc.write_text(mutated)
    libpath = str(tmp_path / f"lib{name}.so")
    oracle.compile_oracle(str(csrc), libpath)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=libpath)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    if r.returncode != 0:
        return  # the mutant crashed the pin run: caught
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED_PINS")]
    assert line, r.stdout + r.stderr
    failed = [x for x in line[0].split(" ", 1)[1].split(",") if x]
    assert failed, f"mutant {name} passed every pin"
