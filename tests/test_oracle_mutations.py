"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign or index, a swapped operand), compiles the copy
and runs every pin against it; at least one pin has to fail.  The shipped
oracle source is never modified.
"""
import os

import pytest

import oracle
from oracle.build import SOURCE, build_oracle
from tests import pins

MUTATIONS = {
    "causal_excludes_self": ("int64_t hi = k_hi < pos + 1 ? k_hi : pos + 1;",
                             "int64_t hi = k_hi < pos ? k_hi : pos;"),
    "wrong_kv_head": ("head / group", "head % hkv"),
    "dropped_softmax_scale": ("        s *= softmax_scale;\n", ""),
    "wrong_in_block_offset": ("size_t off = (size_t)(j % p->bs);",
                              "size_t off = (size_t)((j + 1) % p->bs);"),
    "wrong_block_entry": ("int64_t blk = bt[j / p->bs];",
                          "int64_t blk = bt[(j / p->bs) / 2 * 2];"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "max_not_subtracted": ("double w = exp(scores[j - k_lo] - m);",
                           "double w = exp(scores[j - k_lo]);"),
    "history_offset_dropped": ("int64_t pos = hist + t;", "int64_t pos = t;"),
    "values_read_from_keys": ("out[i] += w * pool_elem(p, 1, bt, j, kvh, i);",
                              "out[i] += w * pool_elem(p, 0, bt, j, kvh, i);"),
    "merge_weight_uses_max": ("double w = exp(lse_parts[s] - total);",
                              "double w = exp(lse_parts[s] - m);"),
    "e4m3_subnormal_exponent": ("v = ldexp((double)m / 8.0, -6);",
                                "v = ldexp((double)m / 8.0, -7);"),
    "ties_away_from_zero": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;",
                            "return f + 1.0;"),
    "fp8_scale_dropped": (" *\n           (double)sc[(size_t)blk * p->hkv + kvh];",
                          ";"),
    "quantize_multiplies": ("volatile float q = x / scale;",
                            "volatile float q = x * scale;"),
    "shard_runs_not_tokens": ("return n <= 1 || (j / k) % n == r;",
                              "return n <= 1 || (j % n) == r;"),
    "shard_off_by_one_rank": ("return n <= 1 || (j / k) % n == r;",
                              "return n <= 1 || (j / k + 1) % n == r;"),
    "rope_sign_swapped": ("double ya = xa * c - xb * s;", "double ya = xa * c + xb * s;"),
    "rope_wrong_partner": ("int b = neox ? i + half : 2 * i + 1;",
                           "int b = neox ? (i + 1) % half + half : 2 * i + 1;"),
    "bf16_ties_up": ("double k = fr > 0.5 ? fl + 1.0 : fr < 0.5 ? fl : (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);",
                     "double k = fr >= 0.5 ? fl + 1.0 : fl;"),
    "e2m1_subnormal_doubled": ("double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                               "double v = e == 0 ? 1.0 * m : ldexp(1.0 + 0.5 * m, e - 1);"),
    "e2m1_exponent_bias": ("double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                           "double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 2);"),
    "e2m1_top_range_step": ("return (uint8_t)(sign | (uint8_t)(round_half_even(0.5 * a) + 4.0));",
                            "return (uint8_t)(sign | (uint8_t)(floor(0.5 * a) + 4.0));"),
    "nvfp4_nibbles_swapped": ("uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
                              "uint8_t code = (i & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    "nvfp4_micro_scale_dropped": ("return pko_e2m1_value(code) * pko_e4m3_value(ms) *",
                                  "return pko_e2m1_value(code) * 1.0 *"),
    "nvfp4_wrong_micro_block": ("uint8_t ms = tile[mo + i / 16];",
                                "uint8_t ms = tile[mo + (i / 16 + 1) % (p->d / 16)];"),
    "nvfp4_groups_ignored": ("int64_t gs = bs < 64 ? bs : 64;", "int64_t gs = bs;"),
    "nvfp4_amax_without_six": ("volatile float six_s = 6.0f * scale;",
                               "volatile float six_s = scale;"),
    "nvfp4_step_without_tile_scale": ("volatile float step = scale * (float)msv;",
                                      "volatile float step = (float)msv;"),
    "v_append_from_k": ("const uint16_t *vs = v_new + ((size_t)t * hkv + h) * d;",
                        "const uint16_t *vs = k_new + ((size_t)t * hkv + h) * d;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(SOURCE).read()
    assert src.count(before) == 1, f"mutation anchor not unique: {name}"
    mutant = tmp_path / f"mutant_{name}.c"
    mutant.write_text(src.replace(before, after))
    so = build_oracle(str(mutant), str(tmp_path / f"libmutant_{name}.so"))
    lib = oracle.load(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
        except ValueError:
            caught.append(pin.__name__ + " (rejected)")
    assert caught, f"no pin caught the planted mistake {name}"
