"""Each plausible mistake planted in a copy of the oracle's source must fail at least one pin.

The copy is compiled on the CPU into a temporary library; the real oracle is untouched.
"""
import os
import tempfile
from pathlib import Path

import pytest

import oracle
import oracle_pins

SRC = Path(oracle.__file__).resolve().parent / "oracle.c"

# (name, exact text in oracle.c, replacement)
MUTANTS = [
    ("relu_dropped", "s > 0.0 ? s : 0.0", "s"),
    ("relu_sign", "s > 0.0 ? s : 0.0", "s < 0.0 ? s : 0.0"),
    ("scale_dropped", "out[r * out_row_stride + p] = scale * weighted;",
     "out[r * out_row_stride + p] = weighted;"),
    ("scale_next_token", "oracle_f32_le(block + scale_region + 4 * i)",
     "oracle_f32_le(block + scale_region + 4 * ((i + 1) % block_size))"),
    ("per_token_rows", "kd[d] = oracle_e4m3_to_double(block[i * head_dim + d]);",
     "kd[d] = oracle_e4m3_to_double(block[i * (head_dim + 4) + d]);"),
    ("extent_short", "int64_t count = seq_len - next_n + t + 1;",
     "int64_t count = seq_len - next_n + t;"),
    ("extent_slot_reversed", "int64_t count = seq_len - next_n + t + 1;",
     "int64_t count = seq_len - t;"),
    ("weights_transposed", "const double wh = (double)weights[r * num_heads + h];",
     "const double wh = (double)weights[(h * rows + r) % (rows * num_heads)];"),
    ("q_head_slot_swapped", "const double *qh = qd + (r * num_heads + h) * head_dim;",
     "const double *qh = qd + ((h % rows) * num_heads + (r % num_heads)) * head_dim;"),
    ("page_index_off", "const int64_t j = p / block_size;", "const int64_t j = (p + 1) / block_size;"),
    ("abs_weight", "weighted += wh * relu;", "weighted += fabs(wh) * relu;"),
    ("e4m3_bias", "ldexp(1.0 + (double)mantissa / 8.0, exponent - 7)",
     "ldexp(1.0 + (double)mantissa / 8.0, exponent - 8)"),
    ("e4m3_subnormal", "ldexp((double)mantissa / 8.0, -6)", "ldexp((double)mantissa / 8.0, -7)"),
    ("e4m3_nan", "if (exponent == 0xF && mantissa == 0x7) return NAN;", ""),
    ("f32_big_endian",
     "uint32_t bits = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |\n                    ((uint32_t)p[3] << 24);",
     "uint32_t bits = (uint32_t)p[3] | ((uint32_t)p[2] << 8) | ((uint32_t)p[1] << 16) |\n                    ((uint32_t)p[0] << 24);"),
    ("padded_128", "return (max_seq_len + 255) / 256 * 256;", "return (max_seq_len + 127) / 128 * 128;"),
    ("width_floor", "return (seq_len + block_size - 1) / block_size;", "return seq_len / block_size;"),
    ("topk_index_desc", "return (a->index > b->index) - (a->index < b->index);",
     "return (a->index < b->index) - (a->index > b->index);"),
    ("topk_ascending", "if (c != 0) return -c;", "if (c != 0) return c;"),
    ("total_order_zero", "if (sa != sb) return sa ? -1 : 1; /* -0 < +0 */", ""),
    ("tie_excludes_nan", "else if (!(s < thr))", "else if (s == thr)"),
    ("candidate_ge", "if (s > thr)\n                ++cand;", "if (s >= thr)\n                ++cand;"),
    ("fit_ignores_tie_room", "(tie <= top_k && cand + tie >= need)", "(cand + tie >= need)"),
    ("fit_ignores_capacity", "fits[r] = cand <= capacity &&", "fits[r] = "),
    ("slot_tie_forward", "return n < top_k ? top_k - 1 - n : -1;", "return n < top_k ? n : -1;"),
    ("slot_cand_unbounded", "if (is_candidate) return n < capacity ? top_k + n : -1;",
     "if (is_candidate) return top_k + n;"),
    ("schedule_truncated", "const int64_t flat = (int64_t)c * total / num_ctas;",
     "const int64_t flat = (int64_t)c * (total / num_ctas);"),
    ("schedule_floor_tiles", "total += (len + tile_tokens - 1) / tile_tokens;",
     "total += len / tile_tokens;"),
    ("e2m1_bias", ": ldexp(1.0 + 0.5 * mantissa, exponent - 1);",
     ": ldexp(1.0 + 0.5 * mantissa, exponent - 2);"),
    ("e2m1_subnormal", "exponent == 0 ? 0.5 * mantissa", "exponent == 0 ? 1.0 * mantissa"),
    ("ue8m0_bias", "ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 126)"),
    ("mx_q_nibbles_swapped",
     "const uint8_t byte = q[rh * row_bytes + d / 2];\n            const uint8_t nibble = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "const uint8_t byte = q[rh * row_bytes + d / 2];\n            const uint8_t nibble = (d % 2 == 1) ? (byte & 0xF) : (byte >> 4);"),
    ("mx_k_nibbles_swapped",
     "const uint8_t byte = block[i * row_bytes + d / 2];\n                    const uint8_t nibble = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "const uint8_t byte = block[i * row_bytes + d / 2];\n                    const uint8_t nibble = (d % 2 == 1) ? (byte & 0xF) : (byte >> 4);"),
    ("mx_k_scale_group16", "oracle_ue8m0_to_double(block[scale_region + i * groups + d / 32])",
     "oracle_ue8m0_to_double(block[scale_region + i * groups + (d / 16) % groups])"),
    ("mx_k_scales_interleaved", "oracle_ue8m0_to_double(block[scale_region + i * groups + d / 32])",
     "oracle_ue8m0_to_double(block[scale_region + (d / 32) * block_size + i])"),
    ("mx_q_scale_dropped",
     "oracle_e2m1_to_double(nibble) * oracle_ue8m0_to_double(q_sf[rh * groups + d / 32]);",
     "oracle_e2m1_to_double(nibble);"),
]


def _compile(name, text):
    src = SRC.read_text()
    old, new = text
    assert src.count(old) >= 1, f"mutant {name}: text not found in oracle.c"
    mutated = src.replace(old, new, 1)
    d = Path(tempfile.mkdtemp(prefix=f"oracle_mut_{name}_"))
    (d / "oracle.c").write_text(mutated)
    return oracle.compile_oracle(d / "oracle.c", d / "liboracle.so", openmp=False)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    lib = oracle.load(_compile(name, (old, new)))
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except Exception:  # any failure of a pin, including a shape mismatch, catches it
            failures.append(check.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
