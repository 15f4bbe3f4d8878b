"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the
CPU, in a temporary directory), builds it, and runs the pin tests of
``test_oracle_pins`` against it: at least one pin has to fail.
"""
import os

import pytest

from oracle import oracle as orc
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(orc.__file__), "moe_oracle.c")

MUTANTS = {
    "q8k_scale_128": ("float s = 127.0f / amax;", "float s = 128.0f / amax;"),
    "q8k_codes_truncated": ("qb[i] = (int8_t)rintf(t);", "qb[i] = (int8_t)t;"),
    "q8k_min_term_dropped": ("bacc += d4 * (double)sc * (double)P - dmin * (double)m * (double)sums[b * (QK / 32) + j];",
                             "bacc += d4 * (double)sc * (double)P;"),
    "q8k_vector_scale_dropped": ("acc += (double)d[b] * bacc;", "acc += bacc;"),
    "q8k_h_not_requantised": ("o[r] = moq_row_dot_q8k(down_e + (long)r * nsb_i * BLK, nsb_i, hq, hd, hs);",
                              "o[r] = moq_row_dot_q8k(down_e + (long)r * nsb_i * BLK, nsb_i, xq, xd, xs);"),
    "q8k_sums_of_wrong_subblock": ("acc += qb[32 * j + i];", "acc += qb[(32 * j + i + 32) % QK];"),
    "nibbles_swapped": ("int q = hi ? (byte >> 4) : (byte & 15);",
                        "int q = hi ? (byte & 15) : (byte >> 4);"),
    "scale_high_bits_shift": ("*sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);",
                              "*sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 2);"),
    "min_high_bits_wrong_byte": ("*m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);",
                                 "*m = (scales[j + 4] >> 4) | ((scales[j - 4] >> 6) << 4);"),
    "min_term_dropped": ("out[i] = d * (double)sc * (double)q - dmin * (double)m;",
                         "out[i] = d * (double)sc * (double)q;"),
    "d_dmin_swapped": ("double d = half_bits_to_double(dbits);",
                       "double d = half_bits_to_double(mbits);"),
    "subnormal_exponent": ("v = ldexp((double)mant, -24);", "v = ldexp((double)mant, -14);"),
    "half_exponent_bias": ("v = ldexp((double)(1024 + mant), expo - 25);",
                           "v = ldexp((double)(1024 + mant), expo - 24);"),
    "chunk_index": ("int c = i / 64;", "int c = (i / 32) % 4;"),
    "silu_sign": ("h[r] = g / (1.0 + exp(-g)) * u;", "h[r] = g / (1.0 + exp(g)) * u;"),
    "silu_on_up": ("h[r] = g / (1.0 + exp(-g)) * u;", "h[r] = u / (1.0 + exp(-u)) * g;"),
    "renorm_dropped": ("w[(long)t * k + j] = pt[idx[(long)t * k + j]] / sel_sum;",
                       "w[(long)t * k + j] = pt[idx[(long)t * k + j]];"),
    "ties_highest_index": ("(best < 0 || pt[e] > pt[best])", "(best < 0 || pt[e] >= pt[best])"),
    "bias_dropped": ("l[e] = acc + (bias ? (double)bias[e] : 0.0);", "l[e] = acc;"),
    "down_row_stride": ("o[r] = row_dot(down_e + (long)r * nsb_i * BLK, I, h, tmp);",
                        "o[r] = row_dot(down_e + (long)r * nsb_h * BLK, I, h, tmp);"),
    "router_weight_ignored": ("yt[i] += wj * o[i];", "yt[i] += o[i];"),
    "permutation_unstable": ("perm[cursor[idx[p]]++] = (int32_t)p;",
                             "perm[cursor[idx[p]]++] = (int32_t)(n - 1 - p);"),
    "gate_up_swapped_in_ffn": ("moq_expert(xv, gate + e * gate_bytes, up + e * gate_bytes,",
                               "moq_expert(xv, up + e * gate_bytes, gate + e * gate_bytes,"),
    "rmsnorm_no_sqrt": ("double inv = 1.0 / sqrt(ss / (double)H + eps);",
                        "double inv = 1.0 / (ss / (double)H + eps);"),
    "rmsnorm_sum_not_mean": ("double inv = 1.0 / sqrt(ss / (double)H + eps);",
                             "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_eps_outside_root": ("double inv = 1.0 / sqrt(ss / (double)H + eps);",
                                 "double inv = 1.0 / (sqrt(ss / (double)H) + eps);"),
    "rmsnorm_gamma_ignored": ("out[(long)t * H + i] = (float)((double)xt[i] * inv * (double)gamma[i]);",
                              "out[(long)t * H + i] = (float)((double)xt[i] * inv);"),
    "residual_dropped": ("out[i] = (double)hidden[i] + y[i];", "out[i] = y[i];"),
    "residual_doubled": ("out[i] = (double)hidden[i] + y[i];",
                         "out[i] = 2.0 * (double)hidden[i] + y[i];"),
}


def _pin_calls(o):
    calls = []
    for blk in pins._golden_blocks():
        calls.append(lambda b=blk: pins.test_hand_built_block(o, b))
    for name in dir(pins):
        fn = getattr(pins, name)
        if not name.startswith("test_") or not callable(fn) or name == "test_hand_built_block":
            continue
        if name == "test_ffn_brute_force_rectangular":
            calls.append(lambda: pins.test_ffn_brute_force_rectangular(o, 512, 256))
            calls.append(lambda: pins.test_ffn_brute_force_rectangular(o, 256, 512))
        else:
            calls.append(lambda f=fn: f(o))
    return calls


def test_unmutated_source_passes_every_pin(tmp_path):
    so = orc.build(force=True, src=SRC, out=str(tmp_path / "liboracle_ref.so"))
    o = orc.Oracle(orc.load_variant(so))
    for call in _pin_calls(o):
        call()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(before, after))
    so = orc.build(force=True, src=str(src), out=str(tmp_path / f"lib_{name}.so"))
    o = orc.Oracle(orc.load_variant(so))
    failures = 0
    for call in _pin_calls(o):
        try:
            call()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin catches the planted mistake {name}"
