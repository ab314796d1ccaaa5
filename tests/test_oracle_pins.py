"""CPU tests: the oracle against its pins, and the pins against planted mistakes."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

from tests import oracle_pins as P

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "moe_oracle.cpp")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle, pin):
    pin(oracle)


# Each mutant is one plausible mistake in the oracle (a dropped term, a wrong
# sign, a swapped or transposed operand, a wrong tie rule, double rounding).
# The pins above must catch every one of them.
MUTANTS = {
    "silu_sign": ("float s = g / (1.0f + std::exp(-g));", "float s = g / (1.0f + std::exp(g));"),
    "gate_up_swapped": ("const uint16_t* wg = w_gate_up_e + (size_t)r * H;",
                        "const uint16_t* wg = w_gate_up_e + (size_t)(I + r) * H;\n"
                        "    const uint16_t* wg_unused = w_gate_up_e + (size_t)r * H; (void)wg_unused;"),
    "tie_to_higher_id": ("if (best < 0 || l[e] > l[best]) best = e;",
                         "if (best < 0 || l[e] >= l[best]) best = e;"),
    "no_renormalisation": ("for (int j = 0; j < K; ++j) w[j] = p[j] / s;\n}\n\nint oracle_topk",
                           "for (int j = 0; j < K; ++j) w[j] = p[j];\n}\n\nint oracle_topk"),
    "double_rounding": ("return oracle_f32_to_bf16(s * u);",
                        "return oracle_f32_to_bf16(oracle_bf16_to_f32(oracle_f32_to_bf16(s)) * u);"),
    "down_transposed": ("const uint16_t* wd = w_down_e + (size_t)j * I;\n    for (int r = 0; r < I; ++r)\n"
                        "      acc = acc + oracle_bf16_to_f32(h_row[r]) * oracle_bf16_to_f32(wd[r]);",
                        "for (int r = 0; r < I; ++r)\n"
                        "      acc = acc + oracle_bf16_to_f32(h_row[r]) * oracle_bf16_to_f32(w_down_e[(size_t)r * H + (j % H)] );"),
    "bias_dropped": ("if (bias) acc = acc + bias[e];", "(void)bias;"),
    "first_slot_weight": ("float ws = routed_scale * w[(size_t)m * K + s];", "float ws = routed_scale * w[(size_t)m * K];"),
    "truncating_round": ("u += 0x7FFFu + lsb;", "(void)lsb;"),
    "router_transposed": ("float wv = oracle_bf16_to_f32(w_router[(size_t)e * H + h]);",
                          "float wv = oracle_bf16_to_f32(w_router[((size_t)h * E + e) % ((size_t)E * H)]);"),
    "softmax_shift_missing_in_sum": ("for (int e = 0; e < E; ++e) z = z + std::exp(l[e] - lmax);",
                                     "for (int e = 0; e < E; ++e) z = z + std::exp(l[e]);"),
    "lm_head_transposed": ("const uint16_t* wr = w + (size_t)v * H;",
                           "const uint16_t* wr = w + ((size_t)v % (size_t)H) * H;"),
    "lm_head_last_term_dropped": ("for (int k = 0; k < H; ++k) acc",
                                  "for (int k = 0; k + 1 < H; ++k) acc"),
    "shared_expert_dropped": ("for (int j = 0; j < H; ++j) acc[j] = acc[j] + ys[j];", "(void)ys;"),
    "routed_scale_ignored": ("float ws = routed_scale * w[(size_t)m * K + s];", "float ws = w[(size_t)m * K + s];"),
    "e4m3_bias_off_by_one": ("mag = std::ldexp(1.0f + (float)m / 8.0f, e - 7);",
                             "mag = std::ldexp(1.0f + (float)m / 8.0f, e - 8);"),
    "fp8_gate_scale_ignored": ("h_out[r] = oracle_swiglu_bf16(s_gu_e[r] * g, s_gu_e[I + r] * u);",
                               "h_out[r] = oracle_swiglu_bf16(g, s_gu_e[I + r] * u);"),
    "fp8_down_scale_shifted": ("y[j] = s_d_e[j] * acc;", "y[j] = s_d_e[(j + 1) % H] * acc;"),
    "selection_weights_from_biased_logits": ("const float* wlog = sel_only ? unbiased.data() : logits.data();",
                                             "const float* wlog = logits.data();"),
}


def _build_mutant(tmpdir, name, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutant {name}: anchor text not found in the oracle"
    msrc = src.replace(old, new, 1)
    path = os.path.join(tmpdir, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(msrc)
    so = os.path.join(tmpdir, f"lib{name}.so")
    from oracle import oracle as O
    subprocess.run(["g++", *O.CXXFLAGS, path, "-o", so], check=True)
    return so


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant_dir, name):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    old, new = MUTANTS[name]
    so = _build_mutant(mutant_dir, name, old, new)
    from oracle.oracle import Oracle
    mut = Oracle(so)
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mut)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
