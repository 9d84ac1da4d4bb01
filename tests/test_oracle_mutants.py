"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Each mutant is a textual edit of ``oracle/oracle.c`` compiled into a
temporary library and checked in a child process (a mutant may crash, which
also counts as caught).  The original snippet must occur exactly once, so
this test fails loudly if the oracle source changes under it.
"""
import json
import os
import subprocess
import sys

import pytest

from oracle.oracle import SOURCE, compile_source

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

MUTANTS = [
    ("diagonal_dropped", "int32_t kb = 0, ke = position + 1;", "int32_t kb = 0, ke = position;"),
    ("gqa_modulo", "h / group, num_heads_kv", "h % num_heads_kv, num_heads_kv"),
    ("scale_dropped", "double s = scale * dot;", "double s = dot;"),
    ("stabiliser_sign", "double w = exp(scores[j - key_begin] - m);",
     "double w = exp(m - scores[j - key_begin]);"),
    ("normalisation_dropped", "o_out[d] /= l;", "o_out[d] /= 1.0;"),
    ("position_ignores_computed", "int32_t position = num_computed[r] + i;",
     "int32_t position = i;"),
    ("slot_ignores_computed", "int64_t position = (int64_t)num_computed[r] + i;",
     "int64_t position = (int64_t)i;"),
    ("slot_block_unscaled", "slot_mapping[first + i] = physical * block_size + offset;",
     "slot_mapping[first + i] = physical + offset;"),
    ("merge_ignores_l", "double w = exp(m_parts[p] - m) * l_parts[p];",
     "double w = exp(m_parts[p] - m);"),
    ("write_value_from_key", "value_cache[slot * row + e] = value[(int64_t)t * row + e];",
     "value_cache[slot * row + e] = key[(int64_t)t * row + e];"),
    ("keys_read_from_values", "const float *kj = k_ctx +", "const float *kj = v_ctx +"),
    ("gather_offset_wrong", "int64_t slot = (int64_t)physical * block_size + j % block_size;",
     "int64_t slot = (int64_t)physical * block_size + (j + 1) % block_size;"),
    ("prefix_length_unchecked", "if ((int64_t)n * block_size > num_computed[r]) return ORACLE_BAD_METADATA;",
     "if (0) return ORACLE_BAD_METADATA;"),
    ("length_identity_unchecked", "if (num_computed[r] + q_len != seq_lens[r]) return ORACLE_BAD_METADATA;",
     "if (0) return ORACLE_BAD_METADATA;"),
    ("e4m3_ties_away", "double v = rint(a / quantum) * quantum;", "double v = round(a / quantum) * quantum;"),
    ("e4m3_no_saturation", "if (v > 448.0) v = 448.0;", "if (0) v = 448.0;"),
    ("e4m3_wrong_bias", "else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("fp8_scale_multiplied", "return (float)bf16_to_double(bits) / scale;", "return (float)bf16_to_double(bits) * scale;"),
    ("fp8_key_scale_dropped", "softmax_scale * k_scale, scores, &m, &l, ov);", "softmax_scale, scores, &m, &l, ov);"),
    ("fp8_value_scale_dropped", "for (int32_t d = 0; d < head_dim; ++d) orow[d] = ov[d] * v_scale;",
     "for (int32_t d = 0; d < head_dim; ++d) orow[d] = ov[d];"),
    ("zero_value_untouched", "memset(value_cache + b * block_bytes, 0, (size_t)block_bytes);", ";"),
    ("zero_wrong_block", "memset(key_cache + b * block_bytes, 0, (size_t)block_bytes);",
     "memset(key_cache + ((b + 1) % num_blocks) * block_bytes, 0, (size_t)block_bytes);"),
    ("zero_negative_ids_wrap", "if (b < 0) continue;", "if (b < 0) b += num_blocks;"),
    ("query_head_transposed", "const uint16_t *qrow = q + ((int64_t)t * num_heads_q + h) * head_dim;",
     "const uint16_t *qrow = q + ((int64_t)t * num_heads_q + (num_heads_q - 1 - h)) * head_dim;"),
]

CHILD = r"""
import json, sys
sys.path[:0] = [sys.argv[2], sys.argv[3]]
from oracle.oracle import Oracle
import oracle_pins
print(json.dumps(oracle_pins.run_all(Oracle(sys.argv[1]))))
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SOURCE, encoding="utf-8").read()
    assert src.count(old) == 1, f"snippet for {name} not found exactly once"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    lib = compile_source(str(mutated), str(tmp_path / "liboracle_mut.so"))
    proc = subprocess.run([sys.executable, "-c", CHILD, lib, ROOT, TESTS],
                          capture_output=True, text=True, timeout=300,
                          env={**os.environ, "OMP_NUM_THREADS": "2"})
    if proc.returncode != 0:
        return  # crashed: caught
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"
