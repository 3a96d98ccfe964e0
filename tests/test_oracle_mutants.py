"""Planted mistakes: each mutant is a copy of the oracle source with one
plausible error (a dropped term, a wrong shift, index or sign, a swapped
operand, a wrong tie-break ...), compiled on the CPU into a temporary
library.  Every mutant must fail at least one pin; otherwise the pins would
not notice that mistake in the real oracle."""
import os
import shutil
import tempfile

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "drop_min_term": [("w[j] = value - min_part;", "w[j] = value;")],
    "swap_scale_min_nibbles": [("int sc = scales[j / 16];",
                                "int sc = ((scales[j / 16] & 15) << 4) | (scales[j / 16] >> 4);")],
    "shift_g_not_2g": [("(qs[32 * h + l] >> (2 * g)) & 3", "(qs[32 * h + l] >> g) & 3")],
    "qs_half_stride_16": [("(qs[32 * h + l] >> (2 * g)) & 3", "(qs[16 * h + l] >> (2 * g)) & 3")],
    "subblock_of_32": [("int sc = scales[j / 16];", "int sc = scales[j / 32];")],
    "half_exponent_bias": [("v = ldexp((double)(1024 + frac), expo - 25);",
                            "v = ldexp((double)(1024 + frac), expo - 24);")],
    "bf16_shift": [("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;")],
    "cb2_nibble_order": [("(sc[group / 2] >> (4 * (group % 2))) & 15",
                          "(sc[group / 2] >> (4 * (1 - group % 2))) & 15")],
    "cb2_ignore_sign": [("w[j] = negate ? -value : value;", "w[j] = value;")],
    "cb2_reversed_entry": [("codebook[8 * idx[o] + b]", "codebook[8 * idx[o] + (7 - b)]")],
    "cb2_group_of_64": [("int group = j / 32;", "int group = j / 64;")],
    "tie_break_higher_id": [("return ia < ib;", "return ia > ib;")],
    "nan_ranks_first": [("(l != l) ? -INFINITY", "(l != l) ? INFINITY")],
    "softmax_no_shift": [("w[i] = exp(rank_value(lg[ids[i]]) - lmax);",
                          "w[i] = exp(rank_value(lg[ids[i]]) - lmax + 0.5 * (i > 0));")],
    "sigmoid_sign": [("w[i] = 1.0 / (1.0 + exp(-rank_value(lg[ids[i]])));",
                      "w[i] = 1.0 / (1.0 + exp(rank_value(lg[ids[i]])));")],
    "offsets_inclusive": [("offsets[e] = run;\n            run += c;",
                           "run += c;\n            offsets[e] = run;")],
    "perm_slot_major": [("for (int t = 0; t < T; ++t)\n                for (int i = 0; i < k; ++i)\n"
                         "                    if (ids[(int64_t)t * k + i] == e) perm[pos++] = t * k + i;",
                         "for (int i = 0; i < k; ++i)\n                for (int t = 0; t < T; ++t)\n"
                         "                    if (ids[(int64_t)t * k + i] == e) perm[pos++] = t * k + i;")],
    "silu_sign": [("h[n] = g / (1.0 + exp(-g)) * u;", "h[n] = g / (1.0 + exp(g)) * u;")],
    "gate_up_swapped": [("h[n] = g / (1.0 + exp(-g)) * u;", "h[n] = u / (1.0 + exp(-u)) * g;")],
    "down_reversed_h": [("acc += (double)rowbuf[n] * h[n];", "acc += (double)rowbuf[n] * h[I - 1 - n];")],
    "combine_wrong_slot_weight": [("yt[m] += w[i] * o[m];", "yt[m] += w[k - 1 - i] * o[m];")],
    "row_blocks_not_advanced": [("orc_q2k_dequant_block(row + (int64_t)b * ORC_Q2K_BYTES, out + b * ORC_QK);",
                                 "orc_q2k_dequant_block(row, out + b * ORC_QK);")],
    "up_reads_gate": [("dequant_row(L, L->format, wu + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);",
                       "dequant_row(L, L->format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);")],
    "min_term_uses_d": [("float min_part = dmin * (float)(sc >> 4);",
                         "float min_part = d * (float)(sc >> 4);")],
    "sigmoid_weights_not_normalised": [
        ("            w[i] = 1.0 / (1.0 + exp(-rank_value(lg[ids[i]])));\n            sum += w[i];\n"
         "        }\n        for (int i = 0; i < k; ++i) w[i] /= sum;",
         "            w[i] = 1.0 / (1.0 + exp(-rank_value(lg[ids[i]])));\n            sum += w[i];\n"
         "        }")],
    "down_expert_stride_of_gate": [("L->w_down + (int64_t)e * L->down_expert_stride",
                                    "L->w_down + (int64_t)e * L->gate_up_expert_stride")],
    "down_row_bytes_of_gate": [("dequant_row(L, L->down_format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);",
                                "dequant_row(L, L->down_format, wd + (int64_t)m * L->gate_up_row_bytes, I, rowbuf);")],
    "down_in_gate_format": [("dequant_row(L, L->down_format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);",
                             "dequant_row(L, L->format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);")],
    "gate_in_down_format": [("dequant_row(L, L->format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);",
                             "dequant_row(L, L->down_format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);")],
    "formats_swapped": [("dequant_row(L, L->format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);",
                         "dequant_row(L, L->down_format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);"),
                        ("dequant_row(L, L->format, wu + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);",
                         "dequant_row(L, L->down_format, wu + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);"),
                        ("dequant_row(L, L->down_format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);",
                         "dequant_row(L, L->format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);")],
    "q2k_three_bit_field": [("(qs[32 * h + l] >> (2 * g)) & 3", "(qs[32 * h + l] >> (2 * g)) & 7")],
    "q2k_halves_swapped": [("(qs[32 * h + l] >> (2 * g)) & 3", "(qs[32 * (1 - h) + l] >> (2 * g)) & 3")],
    "cb2_drops_d": [("float value = d * (float)scale;", "float value = (float)scale;")],
    "cb2_sign_bits_reversed": [("int negate = (sgn[o] >> b) & 1;", "int negate = (sgn[o] >> (7 - b)) & 1;")],
    "cb2_index_per_4": [("int o = j / 8;\n        int b = j % 8;", "int o = j / 4;\n        int b = j % 8;")],
    "route_picks_repeat": [("        ids[i] = best;\n        used[best] = 1;", "        ids[i] = best;")],
    "combine_averages_slots": [("yt[m] += w[i] * o[m];", "yt[m] += w[i] * o[m] / k;")],
    # K-quant formats
    "k4_scale_low_shift": [("*sc = (p[s + 4] & 15) | ((p[s - 4] >> 6) << 4);",
                            "*sc = (p[s + 4] & 15) | ((p[s - 4] >> 6) << 5);")],
    "k4_min_from_scale_byte": [("*m = (p[s + 4] >> 4) | ((p[s] >> 6) << 4);",
                                "*m = (p[s + 4] >> 4) | ((p[s - 4] >> 6) << 4);")],
    "k4_min_mask_5bit": [("*m = p[s + 4] & 63;", "*m = p[s + 4] & 31;")],
    "q4k_nibbles_swapped": [("int q = r < 32 ? (byte & 15) : (byte >> 4);",
                             "int q = r < 32 ? (byte >> 4) : (byte & 15);")],
    "q4k_chunk_stride_64": [("int byte = qs[32 * c + l];\n        int q = r < 32",
                             "int byte = qs[64 * (c / 2) + l];\n        int q = r < 32")],
    "q4k_drops_min": [("        w[j] = value - min_part;\n    }\n}\n\n/* Q5_K",
                       "        w[j] = value;\n    }\n}\n\n/* Q5_K")],
    "q5k_high_bit_by_lane": [("int q = low + 16 * ((qh[l] >> s) & 1);",
                              "int q = low + 16 * ((qh[s] >> (l % 8)) & 1);")],
    "q5k_high_bit_weight_32": [("int q = low + 16 * ((qh[l] >> s) & 1);",
                                "int q = low + 32 * ((qh[l] >> s) & 1);")],
    "q5k_qs_at_16": [("const uint8_t *qs = blk + 48;", "const uint8_t *qs = blk + 16;")],
    "q6k_no_offset": [("int q = low + 16 * high - 32;", "int q = low + 16 * high;")],
    "q6k_ql_half_stride_32": [("int byte = ql[64 * h + 32 * (u & 1) + l];",
                               "int byte = ql[32 * h + 32 * (u & 1) + l];")],
    "q6k_qh_shift_u": [("int high = (qh[32 * h + l] >> (2 * u)) & 3;",
                        "int high = (qh[32 * h + l] >> u) & 3;")],
    "q6k_scale_per_32": [("float scale_part = d * (float)scales[j / 16];",
                          "float scale_part = d * (float)scales[j / 32];")],
    "q6k_unsigned_scales": [("const int8_t *scales = (const int8_t *)(blk + 192);",
                             "const uint8_t *scales = (const uint8_t *)(blk + 192);")],
    "q6k_d_offset": [("float d = (float)orc_half_to_double(rd16(blk + 208));",
                      "float d = (float)orc_half_to_double(rd16(blk + 206));")],
    "mxfp4_nibbles_swapped": [("int code = r < 16 ? (byte & 15) : (byte >> 4);",
                               "int code = r < 16 ? (byte >> 4) : (byte & 15);")],
    "mxfp4_scale_bias_126": [("double scale = e == 255 ? NAN : ldexp(1.0, e - 127);",
                              "double scale = e == 255 ? NAN : ldexp(1.0, e - 126);")],
    "mxfp4_e2m1_six_is_five": [("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}",
                                "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}")],
    "mxfp4_sign_bit_2": [("return (code & 8) ? -v : v;", "return (code & 4) ? -v : v;")],
    "mxfp4_qs_offset_0": [("int byte = b[1 + r % 16];", "int byte = b[r % 16];")],
    "mxfp4_block_stride_16": [("const uint8_t *b = blk + (j / 32) * ORC_MX_BYTES;",
                               "const uint8_t *b = blk + (j / 32) * 16;")],
    "kquant_down_reads_q5k": [("            orc_q6k_dequant_block(row + (int64_t)b * ORC_Q6K_BYTES, out + b * ORC_QK);",
                               "            orc_q5k_dequant_block(row + (int64_t)b * ORC_Q6K_BYTES, out + b * ORC_QK);")],
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="ds4g_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_mutant_patterns_exist():
    src = open(oracle.SOURCE).read()
    for name, edits in MUTANTS.items():
        for old, _ in edits:
            assert src.count(old) >= 1, (name, old)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_dir):
    src = open(oracle.SOURCE).read()
    for old, new in MUTANTS[name]:
        src = src.replace(old, new, 1)
    path = os.path.join(mutant_dir, name + ".c")
    with open(path, "w") as f:
        f.write(src)
    lib = oracle.build(path, os.path.join(mutant_dir, name + ".so"))
    orc = oracle.Oracle(lib)
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failures.append(pin.__name__)
        except (ValueError, FloatingPointError, IndexError):
            failures.append(pin.__name__)
        if failures:
            break
    assert failures, f"planted mistake {name!r} passed every pin"
