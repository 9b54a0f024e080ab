"""Plant one plausible mistake at a time in a copy of the oracle's C source, compile it,
and check that at least one pin fails.  This shows the pins would notice a dropped term,
a wrong index or sign, a transposed operand or a different rounding in the oracle.
Nothing here touches the real oracle or a GPU."""

import os

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("GQA maps head h to h % Hkv", "const int kvh = h / group;", "const int kvh = h % kv_heads;"),
    ("softmax scale dropped", "logits[t - lo] = scale * dot;", "logits[t - lo] = dot;"),
    ("reversed offset inside the block when reading K",
     "int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + i;\n      double dot",
     "int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + (ORACLE_BLOCK_SIZE - 1 - i);\n      double dot"),
    ("pool index transposed (head-major)", "int64_t row = (phys * kv_heads + kvh)",
     "int64_t row = (kvh * num_blocks + phys)"),
    ("first softmax term left unexponentiated",
     "for (int t = lo; t < T; ++t) {\n      logits[t - lo] = exp(", "for (int t = lo + 1; t < T; ++t) {\n      logits[t - lo] = exp("),
    ("last token dropped from the value sum",
     "for (int t = lo; t < T; ++t) {\n      int j = t / ORACLE_BLOCK_SIZE;\n      int i = t % ORACLE_BLOCK_SIZE;\n      int64_t phys = block_tables[(int64_t)b * max_blocks_per_seq + j];\n      int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + i;\n      double w",
     "for (int t = lo; t < T - 1; ++t) {\n      int j = t / ORACLE_BLOCK_SIZE;\n      int i = t % ORACLE_BLOCK_SIZE;\n      int64_t phys = block_tables[(int64_t)b * max_blocks_per_seq + j];\n      int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + i;\n      double w"),
    ("weights not normalised", "double w = logits[t - lo] / denom;", "double w = logits[t - lo];"),
    ("no max shift (overflows on large logits)", "logits[t - lo] = exp(logits[t - lo] - lmax);",
     "logits[t - lo] = exp(logits[t - lo]);"),
    ("bf16 widened with the wrong shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("quantiser divides by 128", "float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    ("quantiser rounds half away from zero", "float r = rintf(y);", "float r = roundf(y);"),
    ("quantiser multiplies by a reciprocal", "float y = x[i] / s;", "float y = x[i] * (1.0f / s);"),
    ("quantiser truncates", "float r = rintf(y);", "float r = truncf(y);"),
    ("INT8 dequantisation ignores the scale", "return (double)scales[row] * (double)p[row * head_dim + c];",
     "return (double)p[row * head_dim + c];"),
    ("cache write offset reversed",
     "int64_t dst = ((block * kv_heads + h) * ORACLE_BLOCK_SIZE + offset) * (int64_t)head_dim;",
     "int64_t dst = ((block * kv_heads + h) * ORACLE_BLOCK_SIZE + (ORACLE_BLOCK_SIZE - 1 - offset)) * (int64_t)head_dim;"),
    ("INT8 write ignores the head", "int64_t srow = (block * kv_heads + h) * ORACLE_BLOCK_SIZE + offset;",
     "int64_t srow = (block * kv_heads + 0) * ORACLE_BLOCK_SIZE + offset;"),
    ("E4M3 decoded with exponent bias 8", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("E4M3 subnormals on the wrong grid", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("E4M3 encode rounds half away from zero", "const double q = rint(ldexp(a, 3 - k));",
     "const double q = round(ldexp(a, 3 - k));"),
    ("E4M3 encode does not saturate", "if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7F;"),
    ("FP8 scale uses the INT8 range", "float s = amax / 448.0f;", "float s = amax / 127.0f;"),
    ("causal limit off by one (query sees its successor)",
     "const int T = context_lens[b] - (num_queries - 1 - qi);",
     "const int T = context_lens[b] - (num_queries - 2 - qi) - (qi == num_queries - 1);"),
    ("queries in reverse order", "const int T = context_lens[b] - (num_queries - 1 - qi);",
     "const int T = context_lens[b] - qi;"),
    ("window one token too wide", "const int lo = (window > 0 && T > window) ? T - window : 0;",
     "const int lo = (window > 0 && T > window) ? T - window - 1 : 0;"),
    ("window ends at the newest token, not at the query", "const int lo = (window > 0 && T > window) ? T - window : 0;",
     "const int lo = (window > 0 && T > window) ? (context_lens[b] - window > 0 ? context_lens[b] - window : 0) : 0;"),
    ("query widened from the wrong head", "const uint16_t* qrow = q + bh * head_dim;",
     "const uint16_t* qrow = q + ((int64_t)b * num_q_heads + (num_q_heads - 1 - h)) * head_dim;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(mutated)
    lib = oracle.build(path, tmp_path / "liboracle_mutant.so", force=True)
    o = oracle.Oracle(lib)
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # noqa: BLE001 -- any failure counts as "caught"
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake: {name}"
