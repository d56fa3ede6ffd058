"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a one-line textual change to a temporary copy of
oracle/moe_oracle.c, compiled with gcc on the CPU. The oracle under oracle/
is never modified. A mutant that every pin accepts would mean the pins cannot
see that kind of mistake.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "nibble_order_reversed": ("(word >> (4 * (j % 8)))", "(word >> (4 * (7 - j % 8)))"),
    "scale_bias_swapped": ("return fmaf(s, q, b);\n}\n\n/* Weight of input column j of one 6-bit",
                           "return fmaf(b, q, s);\n}\n\n/* Weight of input column j of one 6-bit"),
    "bias_dropped": ("return fmaf(s, q, b);\n}\n\n/* Weight of input column j of one 6-bit",
                     "return s * q;\n}\n\n/* Weight of input column j of one 6-bit"),
    "group_index_ignored": ("& 0xFu);\n    float s = bf16_widen(srow[j / ORACLE_GROUP]);",
                            "& 0xFu);\n    float s = bf16_widen(srow[0]);"),
    "six_bit_scale_bias_swapped": ("& 0x3Fu);\n    float s = bf16_widen(srow[j / ORACLE_GROUP]);\n"
                                   "    float b = bf16_widen(brow[j / ORACLE_GROUP]);",
                                   "& 0x3Fu);\n    float b = bf16_widen(srow[j / ORACLE_GROUP]);\n"
                                   "    float s = bf16_widen(brow[j / ORACLE_GROUP]);"),
    "six_bit_group_index_ignored": ("& 0x3Fu);\n    float s = bf16_widen(srow[j / ORACLE_GROUP]);",
                                    "& 0x3Fu);\n    float s = bf16_widen(srow[0]);"),
    "router_bias_dropped": ("if (bias) acc += bias[e];", ""),
    "no_renormalise": ("topk_w[(size_t)t * k + j] = p[topk_idx[(size_t)t * k + j]] / psum;",
                       "topk_w[(size_t)t * k + j] = p[topk_idx[(size_t)t * k + j]];"),
    "tie_to_higher_index": ("if (best < 0 || l[e] > l[best])", "if (best < 0 || l[e] >= l[best])"),
    "silu_sign": ("return z / (1.0f + expf(-z));", "return z / (1.0f + expf(z));"),
    "gate_up_swapped": ("            return silu(g) * u;", "            return silu(u) * g;"),
    "x_index_reversed": ("g = fmaf(dequant_at(gqr, gsr, gbr, d), x[d], g);",
                         "g = fmaf(dequant_at(gqr, gsr, gbr, d), x[D - 1 - d], g);"),
    "combine_rank0_weight": ("acc = fmaf(topk_w[(size_t)t * k + j], y[",
                             "acc = fmaf(topk_w[(size_t)t * k], y["),
    "group_rank_reversed": ("slot_k[pos] = j;", "slot_k[pos] = k - 1 - j;"),
    "offsets_inclusive": ("offsets[e + 1] = offsets[e] + counts[e];",
                          "offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
    "final_round_truncates": ("u += 0x7FFFu + ((u >> 16) & 1u);", ""),
    "final_round_ties_to_odd": ("u += 0x7FFFu + ((u >> 16) & 1u);",
                                "u += 0x7FFFu + (((u >> 16) & 1u) ^ 1u);"),
    "final_round_ties_away": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "gelu_erf_unscaled": ("erff(g * 0.70710678118654752f)", "erff(g)"),
    "gelu_tanh_no_cubic": ("(g + 0.044715f * g * g * g)", "(g + 0.044715f * g * g)"),
    "clamp_gate_below_too": ("float gc = fminf(g, o->limit);",
                             "float gc = fminf(fmaxf(g, -o->limit), o->limit);"),
    "clamp_up_dropped": ("float uc = fminf(fmaxf(u, -o->limit), o->limit);", "float uc = u;"),
    "six_bit_byte_order": ("if (sh > 2) v |= (uint32_t)qrow[byte + 1] << 8;",
                           "if (sh > 2) v = (v << 8) | qrow[byte + 1];"),
    "six_bit_mask": ("float q = (float)((v >> sh) & 0x3Fu);", "float q = (float)((v >> sh) & 0x1Fu);"),
    "six_bit_row_stride": ("const uint8_t *dqr = (const uint8_t *)dq + (size_t)d * (3 * F / 4);",
                           "const uint8_t *dqr = (const uint8_t *)dq + (size_t)d * (F / 2);"),
}


def _build_mutant(name, old, new, tmp):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(text.replace(old, new))
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", path_so,
                    path_c, "-lm"], check=True)
    return path_so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(name, old, new, tmp)
        failed = []
        with oracle.using(so):
            for check in pins.ALL_CHECKS:
                try:
                    check()
                except AssertionError:
                    failed.append(check.__name__)
                except Exception as exc:  # a mutant may also break an invariant loudly
                    failed.append(f"{check.__name__}:{type(exc).__name__}")
        assert failed, f"no pin catches mutant {name}"
