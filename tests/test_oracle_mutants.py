"""Planted mistakes in the oracle must be caught by its pins (no GPU).

Each case compiles a copy of oracle.c with one plausible mistake (a swapped
nibble, a wrong index, a dropped term or sign, a wrong rounding) into a
temporary library, runs every pin against it, and requires at least one pin to
fail. This shows the pins constrain every part of the oracle.
"""
import os

import pytest

import oracle
from oracle import build as obuild
import pins

SRC = os.path.join(os.path.dirname(obuild.__file__), "oracle.c")

# (name, text to replace, replacement, which occurrence (0-based))
MUTANTS = [
    ("nibble_order", "return (k % 2 == 0) ? (b & 0x0Fu) : (b >> 4);",
     "return (k % 2 == 0) ? (b >> 4) : (b & 0x0Fu);", 0),
    ("nvfp4_scale_index", "scales[n * (K / 16) + k / 16]", "scales[n * (K / 16) + k / 32]", 0),
    ("e2m1_sign_dropped", "return s ? -mag : mag;", "return mag;", 0),
    ("e2m1_subnormal", "0.5 * (double)m : ldexp", "1.0 * (double)m : ldexp", 0),
    ("e2m1_exponent_bias", "(int)e - 1);", "(int)e - 2);", 0),
    ("e4m3_bias", "(int)e - 7);", "(int)e - 8);", 0),
    ("e4m3_subnormal", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", 0),
    ("e4m3_nan", "if (e == 15u && m == 7u) return NAN;", "", 0),
    ("f16_bias", "(int)e - 15);", "(int)e - 14);", 0),
    ("bf16_mantissa", "(double)m / 128.0", "(double)m / 256.0", 0),
    ("q5_plane_bit_order", "(q_hi[n * (K / 8) + k / 8] >> (k % 8))",
     "(q_hi[n * (K / 8) + k / 8] >> (7 - k % 8))", 0),
    ("q5_plane_weight", "q |= hb << 4;", "q |= hb << 3;", 0),
    ("q_min_dropped", "return s * q + m;", "return s * q;", 0),
    ("q_group_index", "scale[n * (K / 32) + k / 32]", "scale[n * (K / 32) + k / 16]", 0),
    ("gemv_last_term_dropped", "for (int64_t k = 0; k < K; ++k) {\n                double t = nvfp4_weight",
     "for (int64_t k = 0; k < K - 1; ++k) {\n                double t = nvfp4_weight", 0),
    ("gemv_x_transposed", "orc_bf16(x[m * K + k]);\n                acc += t;",
     "orc_bf16(x[(k * M + m) % (M * K)]);\n                acc += t;", 0),
    ("residual_sign", "if (r) acc += orc_bf16(r[m * N + n]);", "if (r) acc -= orc_bf16(r[m * N + n]);", 0),
    ("global_scale_dropped", "return c * s * g;", "return c * s;", 0),
    ("silu_sign", "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));", 0),
    ("round_ties_away", "nearbyint(ldexp(a, -qexp))", "round(ldexp(a, -qexp))", 0),
    ("round_precision", "int qexp = e - 8;", "int qexp = e - 9;", 0),
    ("route_no_renorm", "for (int i = 0; i < topk; ++i) w[m * topk + i] /= sel;", "", 0),
    ("route_ties_high_id", "if (best < 0 || p[e] > p[best]) best = e;",
     "if (best < 0 || p[e] >= p[best]) best = e;", 0),
    ("moe_gate_up_swapped", "orc_silu(gate[pr * I + i]) * up[pr * I + i]",
     "orc_silu(up[pr * I + i]) * gate[pr * I + i]", 0),
    ("moe_h_not_rounded", "h_bits[pr * I + i] = (uint16_t)orc_bf16_bits(orc_silu(gate[pr * I + i]) * up[pr * I + i]);",
     "h_bits[pr * I + i] = (uint16_t)orc_bf16_bits(orc_silu(gate[pr * I + i]) * up[pr * I + i] * 1.001);", 0),
    ("moe_weight_dropped", "acc += (use_abs ? fabs(ci) : ci) * d;", "acc += d;", 0),
    ("rms_mean_not_divided", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / sqrt(ss + eps)", 0),
    ("rms_eps_dropped", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / sqrt(ss / (double)K)", 0),
    ("rms_no_root", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / (ss / (double)K + eps)", 0),
    ("rms_gamma_dropped", "orc_bf16(x[m * K + k]) * rm * orc_bf16(gamma[k]);", "orc_bf16(x[m * K + k]) * rm;", 0),
    ("rms_gamma_reversed", "orc_bf16(x[m * K + k]) * rm * orc_bf16(gamma[k]);",
     "orc_bf16(x[m * K + k]) * rm * orc_bf16(gamma[K - 1 - k]);", 0),
    ("moe_down_expert_index", "int64_t e = ids[m * topk + i];\n                const uint8_t* c = dn_codes",
     "int64_t e = ids[m * topk];\n                const uint8_t* c = dn_codes", 0),
]


def _mutate(text, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    assert src.count(old) >= occ + 1, f"mutation pattern for {name} not found"
    mut = tmp_path / f"oracle_{name}.c"
    mut.write_text(_mutate(src, old, new, occ))
    lib = obuild.build(str(mut), str(tmp_path / f"lib_{name}.so"))
    prev = oracle.use_library(lib)
    failed = []
    try:
        for pin in pins.PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    finally:
        oracle.use_library(None)
    assert failed, f"no pin caught the planted mistake {name}"
