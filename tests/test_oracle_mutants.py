"""Planted mistakes in copies of the oracle source must each fail a pin.

Every mutant below is a plausible slip (a dropped term, a wrong index, a
swapped operand, a wrong bias) applied to a private copy of the C oracle and
compiled with gcc on the CPU; the pin battery must reject it.  The real
oracle must pass the same battery.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "gqa_head_modulo": ("int h = i / group;", "int h = i % num_kv_heads;"),
    "scale_dropped": ("z[t] = scale * acc;", "z[t] = acc;"),
    "max_not_subtracted": ("z[t] = exp(z[t] - zmax);", "z[t] = exp(z[t]);"),
    "block_offset_swapped": (
        "int64_t row = (((int64_t)b * block_size + t % block_size) * num_kv_heads + h) * head_dim;\n"
        "                double acc",
        "int64_t row = (((int64_t)b * block_size + t / block_size) * num_kv_heads + h) * head_dim;\n"
        "                double acc"),
    "logical_block_index": (
        "int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];\n"
        "                if (b < 0",
        "int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t % max_blocks_per_seq];\n"
        "                if (b < 0"),
    "last_token_dropped": ("for (int t = 0; t < n; ++t) {\n                int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];\n                if (b < 0",
                           "for (int t = 0; t < n - 1 + (n == 1); ++t) {\n                int32_t b = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];\n                if (b < 0"),
    "heads_dims_transposed": ("* num_kv_heads + h) * head_dim;\n                double acc",
                              "* head_dim + h) * num_kv_heads;\n                double acc"),
    "not_normalised": ("double w = z[t] / denom;", "double w = z[t];"),
    "q_k_swapped_v": ("o[d] += w * decode(dtype, v_cache[row + d]);",
                      "o[d] += w * decode(dtype, k_cache[row + d]);"),
    "f16_bias": ("mag = ldexp((double)(1024 + frac), expo - 25);",
                 "mag = ldexp((double)(1024 + frac), expo - 24);"),
    "f16_subnormal": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    "bf16_implicit_bit": ("mag = ldexp((double)(128 + frac), expo - 134);",
                          "mag = ldexp((double)frac, expo - 134);"),
    "slot_offset": ("slot_mapping[s] = (int64_t)b * block_size + p % block_size;",
                    "slot_mapping[s] = (int64_t)b * block_size + p / block_size;"),
    "slot_position_len": ("int p = n - 1;", "int p = n;"),
    "write_padding_not_skipped": ("if (slot < 0) continue;", "if (slot < 0) slot = 0;"),
    "write_v_into_k": ("memcpy(v_cache + dst, v_new", "memcpy(k_cache + dst, v_new"),
    "copy_v_not_copied": ("memcpy(v_cache + dst[i] * blk, v_cache + src[i] * blk",
                          "memcpy(v_cache + src[i] * blk, v_cache + src[i] * blk"),
    "copy_half_block": ("memcpy(k_cache + dst[i] * blk, k_cache + src[i] * blk, (size_t)blk * 2);",
                        "memcpy(k_cache + dst[i] * blk, k_cache + src[i] * blk, (size_t)blk);"),
    "prefill_rows_not_packed": ("int64_t qrow = (int64_t)cu_q_lens[s] + r;",
                                "int64_t qrow = (int64_t)s + r;"),
    "prefill_gqa_head_modulo": (
        "int h = i / group;\n                for (int d = 0; d < head_dim; ++d) { qd[d] = decode(dtype, qi[d]); o[d] = 0.0; }",
        "int h = i % num_kv_heads;\n                for (int d = 0; d < head_dim; ++d) { qd[d] = decode(dtype, qi[d]); o[d] = 0.0; }"),
    "prefill_max_not_subtracted": (
        "for (int t = 0; t <= p; ++t) { z[t] = exp(z[t] - zmax); denom += z[t]; }",
        "for (int t = 0; t <= p; ++t) { z[t] = exp(z[t]); denom += z[t]; }"),
    "prefill_not_causal": ("int p = n - rows + r;", "int p = n - 1;"),
    "prefill_position_off_by_one": ("int p = n - rows + r;", "int p = n - rows + r - 1 + (r == 0);"),
}


def test_real_oracle_passes_every_pin():
    assert oracle_pins.failing_pins(oracle.default()) == []


_CHILD = """
import json, sys
sys.path[:0] = [{tests!r}, {root!r}]
import oracle, oracle_pins
src = open({src!r}).read()
o = oracle.Oracle(oracle.build(force=True, src={src!r}, out={so!r}))
print(json.dumps(oracle_pins.failing_pins(o)))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    src_path = tmp_path / "oracle_mutant.c"
    src_path.write_text(mutated)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(tests=tests_dir, root=os.path.dirname(tests_dir), src=str(src_path),
                         so=str(tmp_path / "liboracle_mutant.so"))
    # a child process, so that a mutant which reads out of bounds cannot take the suite down
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, f"mutant {name!r} crashed the pin battery: {r.stderr[-400:]}"
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"planted mistake {name!r} passed every pin"
