"""Plant plausible mistakes in copies of the oracle and check the pins catch each one.

Each mutation is a textual edit of the oracle's C source (a dropped term, a wrong
sign, a wrong index or stride, a transposed operand, an off-by-one mask). The
mutated copy is compiled into a temporary library on the CPU; at least one pin
from ``oracle_pins`` must fail on it. The real oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

MUTATIONS = [
    # (name, search, replace, pins that should catch it)
    ("diagonal_dropped", "t2 <= t; t2++", "t2 < t; t2++", oracle_pins.TRIMUL_PINS),
    ("key_read_from_value", "h * HS + C;", "h * HS + 2 * C;", oracle_pins.TRIMUL_PINS),
    ("key_read_from_query", "h * HS + C;", "h * HS;", oracle_pins.TRIMUL_PINS),
    ("scale_multiplied", "dst[t2] = acc / root_hs", "dst[t2] = acc * root_hs", oracle_pins.TRIMUL_PINS),
    ("scale_of_C", "sqrt((double)HS)", "sqrt((double)C)", oracle_pins.TRIMUL_PINS),
    ("scale_missing", "dst[t2] = acc / root_hs", "dst[t2] = acc", oracle_pins.TRIMUL_PINS),
    ("dot_drops_last_term", "d < HS; d++", "d < HS - 1; d++", oracle_pins.TRIMUL_PINS),
    ("query_row_stride", "query = qkv + b * T * C3 + t * C3", "query = qkv + b * T * C3 + t * C",
     oracle_pins.TRIMUL_PINS),
    ("query_head_stride", "query = qkv + b * T * C3 + t * C3 + h * HS",
     "query = qkv + b * T * C3 + t * C3 + h", oracle_pins.TRIMUL_PINS),
    ("batch_ignored_in_key", "key = qkv + b * T * C3 + t2 * C3", "key = qkv + t2 * C3",
     oracle_pins.TRIMUL_PINS),
    ("mask_starts_late", "t2 = t + 1; t2 < T", "t2 = t + 2; t2 < T", oracle_pins.TRIMUL_PINS),
    ("mask_sign", "-INFINITY : NAN", "INFINITY : NAN", oracle_pins.TRIMUL_PINS),
    ("mask_is_zero", "-INFINITY : NAN", "-INFINITY : 0.0", oracle_pins.TRIMUL_PINS),
    ("row_order_swapped", "const int64_t t = r % T;\n        const int64_t h = (r / T) % NH;",
     "const int64_t h = r % NH;\n        const int64_t t = (r / NH) % T;", oracle_pins.TRIMUL_PINS),
    ("dense_transposed_w", "W[j * I + k]", "W[k * H + j]", oracle_pins.DENSE_PINS),
    ("dense_drops_last_k", "k < I; k++", "k < I - 1; k++", oracle_pins.DENSE_PINS),
    ("dense_sign", "dst[j] = acc;", "dst[j] = -acc;", oracle_pins.DENSE_PINS),
    ("bmm_drops_last_term", "l < D; l++)", "l < D - 1; l++)", oracle_pins.BMM_PINS),
    ("bmm_sign", "y[k] = acc;", "y[k] = -acc;", oracle_pins.BMM_PINS),
    ("bmm_rows_reversed", "x = X + (i * T1 + j) * D", "x = X + (i * T1 + (T1 - 1 - j)) * D",
     oracle_pins.BMM_PINS),
    ("bmm_batch_ignored_in_w", "w = W + (i * T2 + k) * D", "w = W + k * D", oracle_pins.BMM_PINS),
    ("softmax_no_max_subtracted", "if (dst[t2] > m)\n            m = dst[t2];",
     "if (dst[t2] > m)\n            m = 0.0;", oracle_pins.SOFTMAX_PINS),
    ("softmax_min_subtracted", "if (dst[t2] > m)", "if (dst[t2] < m)", oracle_pins.SOFTMAX_PINS),
    ("softmax_sum_drops_diagonal", "t2 <= t; t2++) {\n        dst[t2] = exp",
     "t2 < t; t2++) {\n        dst[t2] = exp", oracle_pins.SOFTMAX_PINS),
    ("softmax_multiplies", "dst[t2] /= sum", "dst[t2] *= sum", oracle_pins.SOFTMAX_PINS),
    ("softmax_upper_not_zero", "dst[t2] = 0.0;\n}", "dst[t2] = 1e-30;\n}", oracle_pins.SOFTMAX_PINS),
    ("softmax_counts_terms", "sum += dst[t2];", "sum += 1.0;", oracle_pins.SOFTMAX_PINS),
    ("f32_diagonal_dropped", "t2 <= t; t2++) {\n        const float *key", "t2 < t; t2++) {\n        const float *key",
     oracle_pins.TRIMUL_F32_PINS),
    ("f32_key_read_from_value", "const float *key = qkv + b * T * C3 + t2 * C3 + h * HS + C;",
     "const float *key = qkv + b * T * C3 + t2 * C3 + h * HS + 2 * C;", oracle_pins.TRIMUL_F32_PINS),
    ("f32_key_read_from_query", "acc += (double)query[d] * (double)key[d];",
     "acc += (double)query[d] * (double)query[d];", oracle_pins.TRIMUL_F32_PINS),
    ("f32_scale_by_hs", "acc += (double)query[d] * (double)key[d];\n        dst[t2] = acc / root_hs;",
     "acc += (double)query[d] * (double)key[d];\n        dst[t2] = acc / (double)HS;", oracle_pins.TRIMUL_F32_PINS),
    ("f32_batch_ignored", "const float *query = qkv + b * T * C3 + t * C3 + h * HS;",
     "const float *query = qkv + t * C3 + h * HS;", oracle_pins.TRIMUL_F32_PINS),
    ("f32_input_rounded_to_bf16", "acc += (double)query[d] * (double)key[d];",
     "acc += (double)(float)(__bf16)query[d] * (double)(float)(__bf16)key[d];", oracle_pins.TRIMUL_F32_PINS),
    ("dense_bf16_truncated", "(uint32_t)h << 16", "((uint32_t)h << 16) & 0xFFFE0000u",
     oracle_pins.ALL_PINS),
]


def _mutated(tmp_path, name, search, replace):
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(search) >= 1, f"mutation {name}: pattern not found in oracle source"
    src = src.replace(search, replace)
    path = os.path.join(str(tmp_path), f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    lib = oracle.compile_oracle(path, os.path.join(str(tmp_path), f"lib{name}.so"), force=True)
    return oracle.Oracle(lib)


@pytest.mark.parametrize("name,search,replace,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, name, search, replace, pins):
    o = _mutated(tmp_path, name, search, replace)
    caught = []
    for pin in pins:
        try:
            pin(o)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutation {name}"
