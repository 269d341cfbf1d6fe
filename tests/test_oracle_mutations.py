"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source, plants one plausible mistake (a dropped
term, a wrong sign or index, a transposed operand, a wrong alignment), builds
the copy with gcc into a temporary directory and runs every pin against it. The
test passes only if at least one pin fails for that mistake. The planted copies
live in pytest's temporary directory; the real oracle is never modified. CPU only.
"""
import os

import pytest

import oracle
import oracle_pins

MUTATIONS = {
    "causal_top_left": ("if (causal && j > i + causal_offset)", "if (causal && j > i)"),
    "kv_head_modulo": ("const int g = h / group;", "const int g = h % Hkv;"),
    "scale_dropped": ("double sij = scale * dot;", "double sij = dot;"),
    "mask_sign": ("if (additive) sij += (double)mask", "if (additive) sij -= (double)mask"),
    "mask_ignores_batch": ("mask[((size_t)b * Sq + i) * Sk + j]", "mask[((size_t)0 * Sq + i) * Sk + j]"),
    "lse_drops_max": ("lse[(size_t)s * rows + r] = m + log(l);", "lse[(size_t)s * rows + r] = log(l);"),
    "no_max_subtraction": ("srow[j] = exp(srow[j] - m);", "srow[j] = exp(srow[j]);"),
    "no_normalisation": ("double pij = srow[j] / l;", "double pij = srow[j];"),
    "keys_reversed": ("dot += qd[d] * kd[j * D + d];", "dot += qd[d] * kd[(Sk - 1 - j) * D + d];"),
    "v_transposed": ("orow[d] += pij * vd[j * D + d];", "orow[d] += pij * vd[d * Sk + j];"),
    "query_head_fixed": ("qd[d] = widen(q[(((size_t)b * Sq + i) * Hq + h) * D + d], dtype);",
                         "qd[d] = widen(q[(((size_t)b * Sq + i) * Hq + 0) * D + d], dtype);"),
    "max_pass_dropped": ("if (sij > m) m = sij;", ";"),
    "bf16_shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "f16_bias": ("expo - 25);", "expo - 24);"),
    "default_scale_sqrt_missing": ("scale = 1.0 / sqrt((double)D);", "scale = 1.0 / (double)D;"),
    "rope_rotation_sign": ("x[2 * i] = x0 * c - x1 * s;", "x[2 * i] = x0 * c + x1 * s;"),
    "rope_frequency_exponent": ("pow(base, -2.0 * i / D)", "pow(base, -1.0 * i / D)"),
    "rope_query_position": ("rope_rotate(qd, D, q_pos0 + i, rope_base, rope_round, dtype);",
                            "rope_rotate(qd, D, k_pos0 + i, rope_base, rope_round, dtype);"),
    "rope_round_truncates": ("nearbyint(x / ulp) * ulp", "trunc(x / ulp) * ulp"),
    "rope_round_types_swapped": ("const int bits = dtype == ORACLE_DTYPE_F16 ? 11 : 8;",
                                 "const int bits = dtype == ORACLE_DTYPE_F16 ? 8 : 11;"),
    "rope_round_skips_keys": ("rope_rotate(kd + j * D, D, k_pos0 + j, rope_base, rope_round, dtype);",
                              "rope_rotate(kd + j * D, D, k_pos0 + j, rope_base, 0, dtype);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(str(path), str(tmp_path / "libmutant.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
        except ValueError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
