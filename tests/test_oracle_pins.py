"""The oracle against what the mathematics fixes (CPU only).

Every pin in ``oracle_pins.py`` must hold for the real oracle, and every
planted mistake below (made in a copy of the oracle's C source, compiled on
the CPU) must trip at least one pin.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins as pins

_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
v = oracle.compile_variant(open({src!r}).read(), {work!r})
caught = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(v)
    except AssertionError:
        caught.append(pin.__name__)
print("CAUGHT", caught)
sys.exit(3 if caught else 0)
"""


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_mod):
    pin(oracle_mod)


# (name, text in mla_oracle.c, replacement): plausible slips, each of which
# must be caught by at least one pin.
MUTATIONS = [
    ("causal_off_by_one", "ctx - sq + i + 1", "ctx - sq + i"),
    ("value_reads_wrong_dims",
     "o[d] += w * cache_elem(cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, j, d);",
     "o[d] += w * cache_elem(cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, j, d + 64);"),
    ("page_and_slot_swapped",
     "int64_t page = bt[(int64_t)b * bt_stride + j / page_size];\n  int64_t slot = j % page_size;",
     "int64_t page = bt[(int64_t)b * bt_stride + j % page_size];\n  int64_t slot = j / page_size;"),
    ("softmax_scale_dropped", "z[j - lo] = scale * acc;", "z[j - lo] = acc;"),
    ("lse_in_log2", "l = m + log(sum);", "l = m + log2(sum);"),
    ("fp8_scale_dropped", "* kv_scale;\n}", ";\n}"),
    ("e4m3_bias_8", "expo - 7);", "expo - 8);"),
    ("e4m3_subnormal_as_normal", "ldexp((double)mant / 8.0, 1 - 7)", "ldexp(1.0 + (double)mant / 8.0, 1 - 7)"),
    ("merge_weight_unnormalised", "w = exp(ls - L);", "w = exp(ls);"),
    ("score_sign_flipped", "acc += mla_oracle_bf16_to_double(q_row[d]) *", "acc -= mla_oracle_bf16_to_double(q_row[d]) *"),
    ("query_row_transposed", "(((int64_t)bb * Sq + i) * H + h)", "(((int64_t)bb * H + h) * Sq + i)"),
    ("bf16_wrong_half", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("weights_skip_max", "double w = exp(z[j - lo] - l);", "double w = exp(z[j - lo] - m);"),
    ("row_query_transposed", "q + (((int64_t)b * Sq + i) * H + h) * ORACLE_D_QK",
     "q + (((int64_t)b * H + h) * Sq + i) * ORACLE_D_QK"),
    ("row_sees_all_tokens_keys", "int64_t n = visible_keys(seq_lens[b], Sq, i, causal);",
     "int64_t n = visible_keys(seq_lens[b], Sq, Sq - 1, causal);"),
    ("epilogue_rope_from_latent", "dst[512 + d] = q_pe[((int64_t)t * H + h) * 64 + d];",
     "dst[512 + d] = ql_nope[((int64_t)t * H + h) * 512 + d];"),
    ("epilogue_page_offset_swapped", "page = slot / page_size;\n      off = slot % page_size;",
     "page = slot % page_size;\n      off = slot / page_size;"),
    ("epilogue_scale_multiplied", "mla_oracle_bf16_to_double(x) / (double)kv_scale",
     "mla_oracle_bf16_to_double(x) * (double)kv_scale"),
    ("encode_ties_to_odd", "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("encode_no_saturation", "if (a > 448.0) return (uint8_t)(sign | 0x7E);",
     "if (a > 448.0) return 0x7F;"),
    ("encode_sign_dropped", "return (uint8_t)(sign | best);", "return (uint8_t)best;"),
    ("gkv_head_stride", "const uint16_t* w = W + ((int64_t)h * 256 + o) * 512;",
     "const uint16_t* w = W + ((int64_t)o * H + h) * 512;"),
    ("gkv_key_value_swapped", "if (o < 128)\n            k[", "if (o >= 128)\n            k["),
    ("gkv_rope_from_latent", "k[(t * H + h) * 192 + 128 + d] = c[512 + d];",
     "k[(t * H + h) * 192 + 128 + d] = c[d];"),
    ("gkv_rows_reversed", "int64_t t = (int64_t)cu_seqlens[b] + j;",
     "int64_t t = (int64_t)cu_seqlens[b + 1] - 1 - j;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests_dir), tests=tests_dir,
                          src=str(mutant), work=str(tmp_path))
    # A separate process: a planted indexing slip may read out of bounds and
    # crash, which also counts as caught.
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"no pin caught the planted mistake {name}: {r.stdout}{r.stderr}"
