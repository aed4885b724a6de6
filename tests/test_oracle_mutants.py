"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of the oracle's C source (on the
CPU, in a temporary directory), builds it, and requires that at least one pin
of ``oracle_pins`` fails on it. Mutations are chosen to stay in bounds, so a
broken copy computes wrong values rather than crashing.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "drop_k_scale": [("* (double)ks;", ";")],
    "drop_q_scale": [("* (double)q_scale[h];", ";")],
    "drop_head_weight": [("total += (double)w[h] * (", "total += (")],
    "no_relu": [("(dot > 0.0 ? dot : 0.0)", "dot")],
    "drop_softmax_scale": [("softmax_scale * head_norm * total", "head_norm * total")],
    "reversed_k_dims": [("dot += qd[h][d] * kd[d];", "dot += qd[h][d] * kd[ORA_DIM - 1 - d];")],
    "causal_excludes_self": [("int64_t n = positions[t] + 1;", "int64_t n = positions[t] > 0 ? positions[t] : 1;")],
    "ignore_page_index": [("(int64_t)bt_row[s / ORA_BLOCK] * ORA_BLOCK", "(int64_t)bt_row[0] * ORA_BLOCK")],
    "interleaved_slots": [("*k_byte = page * page_bytes + off * row;", "*k_byte = slot * (row + 4);"),
                          ("*scale_byte = page * page_bytes + ORA_BLOCK * row + off * 4;",
                           "*scale_byte = slot * (row + 4) + row;")],
    "scale_rounds_down": [("return (float)ldexp(1.0, e);", "return (float)ldexp(1.0, e - 1);")],
    "no_amax_floor": [("if (!(amax >= 1e-10f)) amax = 1e-10f;", "")],
    "ties_away_from_zero": [("q = nearbyint(a / quantum);", "q = round(a / quantum);")],
    "saturate_to_nan": [("if (a >= 448.0) return sign | 0x7E;", "if (a > 448.0) return sign | 0x7F;")],
    "zero_loses_sign": [("if (a == 0.0) return sign;", "if (a == 0.0) return 0;")],
    "subnormal_as_normal": [("if (e < -6) e = -6;", "")],
    "topk_ties_high_index": [("return (i < j) ? -1 : (i > j);", "return (i > j) ? -1 : (i < j);")],
    "schedule_offset_off_by_one": [("int v = l - offset + 1;", "int v = l - offset;")],
    "schedule_no_char_check": [("if (pattern[l] != 'F' && pattern[l] != 'S') return -1;", "")],
    "convert_ignores_stride": [("row[id / block_size] * block_stride_rows", "row[id / block_size] * block_size")],
    "rope_interleaved_pairs": [("x2 = bf16_value(xr[i + ORA_ROPE / 2]);", "x2 = bf16_value(xr[i ^ 1]);")],
    "rope_sine_sign": [("yr[i] = bf16_round(a - b);", "yr[i] = bf16_round(a + b);")],
    "rope_cos_sin_swapped": [("const float c = cos_sin[p * ORA_ROPE + i], s = cos_sin[p * ORA_ROPE + ORA_ROPE / 2 + i];",
                              "const float s = cos_sin[p * ORA_ROPE + i], c = cos_sin[p * ORA_ROPE + ORA_ROPE / 2 + i];")],
    "rope_token_of_row": [("const int64_t p = positions[r / rows_per_token];", "const int64_t p = positions[r % rows_per_token];")],
    "rope_truncates": [("  u += 0x7FFFu + ((u >> 16) & 1u);\n", "")],
    "gather_row_stride_ignored": [("rows + (int64_t)id * row_stride", "rows + (int64_t)id * row_bytes")],
    "gather_keeps_stale_rows": [("        memset(dst, 0, (size_t)row_bytes);\n", "")],
    "e2m1_ties_away_from_zero": [("steps = nearbyint(a / quantum);", "steps = round(a / quantum);")],
    "e2m1_no_saturation": [("if (a >= 6.0) return sign | 0x7;", "")],
    "e2m1_subnormal_dropped": [("if (steps < 2.0) return sign | 0x1;", "if (steps < 2.0) return sign;")],
    "e2m1_exponent_bias_2": [("ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)")],
    "e2m1_scale_uses_fp8_max": [("return ue8m0_of(amax, 6.0f);", "return ue8m0_of(amax, 448.0f);")],
    "fp4_nibbles_swapped": [("(ora_e2m1_encode(x[i] / s) | (ora_e2m1_encode(x[i + 1] / s) << 4))",
                             "(ora_e2m1_encode(x[i + 1] / s) | (ora_e2m1_encode(x[i] / s) << 4))")],
    "fp4_decode_high_nibble_first": [("(4 * (d & 1))", "(4 * (1 - (d & 1)))")],
    # FP4 pages pitched without their scale block (4096 instead of 4352 bytes);
    # a smaller pitch keeps every write inside the cache
    "fp4_page_pitch_without_scales": [
        ("int64_t page_bytes = (fmt == ORA_FMT_FP4) ? ORA_FP4_PAGE_BYTES : ORA_PAGE_BYTES;",
         "int64_t page_bytes = (fmt == ORA_FMT_FP4) ? ORA_BLOCK * ORA_DIM / 2 : ORA_PAGE_BYTES;")],
    "fp4_row_read_as_fp8": [("double v = (fmt == ORA_FMT_FP4) ?", "double v = 0 ?")],
    "convert_counts_padding": [("        ++valid;\n", ""), ("        physical[t * topk + j] = -1;\n",
                                                        "        physical[t * topk + j] = -1;\n        ++valid;\n")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(oracle.SOURCE).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(src)
    lib = oracle.compile_source(path, os.path.join(tmp_path, f"libmut_{name}.so"))
    ora = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(ora)
        except (AssertionError, ValueError, RuntimeError):
            failed.append(pin.__name__)
            break
    assert failed, f"no pin catches mutant {name}"
