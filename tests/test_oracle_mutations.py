"""The oracle's pins are sensitive: plant one plausible mistake at a time in a copy of
the oracle source (on the CPU), rebuild it, and check that at least one pin fails.

A pin that passes on a mutated oracle proves nothing; this file shows that each
class of slip named in the pins' docstring -- a dropped term, a wrong sign, a
wrong index, a transposed operand -- is caught.
"""
import os

import pytest

import tests.test_oracle_pins as pins
from oracle import prism_oracle

SRC = prism_oracle._SRC

# (name, text in the oracle source, replacement)
MUTATIONS = [
    ("delta sign", "al * (S[(size_t)i * dk + j] - be * Sk[i] * kt[j])",
     "al * (S[(size_t)i * dk + j] + be * Sk[i] * kt[j])"),
    ("decay dropped", "S[(size_t)i * dk + j] = al * (", "S[(size_t)i * dk + j] = 1.0 * ("),
    ("decay also on the write", "+ be * vt[i] * kt[j];", "* 1.0 + al * be * vt[i] * kt[j];"),
    ("state read along the wrong axis", "s += S[(size_t)i * dk + j] * kt[j];",
     "s += S[(size_t)j * dk + i] * kt[j];"),
    ("readout with the key", "s += S[(size_t)i * dk + j] * qt[j];", "s += S[(size_t)i * dk + j] * kt[j];"),
    ("conv taps reversed", "acc += w[j * dv + c] * v[(size_t)(t - j) * dv + c];",
     "acc += w[(3 - j) * dv + c] * v[(size_t)(t - j) * dv + c];"),
    ("conv excludes current token", "for (int j = 0; j < 4; ++j)\n                if (t - j >= 0)",
     "for (int j = 1; j < 4; ++j)\n                if (t - j >= 0)"),
    ("gain without the h phi term", "g[c] = Phi + acc * phi;", "g[c] = Phi;"),
    ("residual with Phi instead of GELU", "e[c] = vt[c] - acc * Phi;", "e[c] = vt[c] - Phi;"),
    ("eta slot shifted", "eta[(size_t)t * R + (l - 1)]", "eta[(size_t)t * R + l]"),
    ("gamma slot shifted", "gamma[(size_t)t * R + (l - 1)]", "gamma[(size_t)t * R + (R - l)]"),
    ("chain sign", "r[i] *= (1.0 - et * g[i]);", "r[i] *= (1.0 + et * g[i]);"),
    ("chain without gain", "double x = gm * g[i] * r[i];", "double x = gm * r[i];"),
    ("direction slot shifted", "ul = u + ((size_t)t * R + (l - 1)) * dk;", "ul = u + ((size_t)t * R + (R - l)) * dk;"),
    ("history in reverse order", "vh[(size_t)(3 + t - j) * dv + c]", "vh[(size_t)(j - t - 1) * dv + c]"),
    ("history ignored", "else if (vh) acc +=", "else if (0) acc +="),
    ("initial state ignored", "    if (a->S_init)\n", "    if (0)\n"),
    ("non-linear step adds", "r[i] -= delta;", "r[i] += delta;"),
    ("non-linear step with Phi", "const double delta = z * 0.5 * (1.0 + erf(z * inv_sqrt2));",
     "const double delta = 0.5 * (1.0 + erf(z * inv_sqrt2));"),
    ("gain slot shifted", "pg + ((size_t)t * R + (l - 1)) * dv", "pg + ((size_t)t * R + (R - l)) * dv"),
    ("non-linear factor without gamma", "x = gm * delta;", "x = delta;"),
    ("readout dropped", "        /* readout from the post-update state */",
     "        /* readout from the post-update state */\n        if (0)"),
]


def _pin_suite(mod):
    """Run every pin against `mod`; return the names of the pins that failed."""
    failed = []
    cases = [
        ("gdn", lambda: pins.test_gdn_degenerate_equals_delta_rule(mod)),
        ("gelu", lambda: pins.test_gain_and_residual_match_library_gelu(mod)),
        ("impulse", lambda: pins.test_anchor_impulse_response(mod)),
        ("chain", lambda: pins.test_residual_chain_closed_form(mod)),
        ("brute1", lambda: pins.test_brute_force_transition_products(mod, 1)),
        ("brute4", lambda: pins.test_brute_force_transition_products(mod, 4)),
        ("zero", lambda: pins.test_zero_write_gates_give_zero_state(mod)),
        ("recall", lambda: pins.test_exact_recall_with_orthonormal_keys(mod)),
        ("linattn", lambda: pins.test_no_forget_no_delta_is_causal_linear_attention(mod)),
        ("zeroconv", lambda: pins.test_zero_conv_gives_half_gain(mod)),
        ("inert", lambda: pins.test_history_equals_prepended_inert_tokens(mod)),
        ("split", lambda: pins.test_split_calls_with_history_and_state(mod, (2, 3, 29))),
        ("nl_zero", lambda: pins.test_nonlinear_zero_gain_is_gdn(mod)),
        ("nl_small", lambda: pins.test_nonlinear_small_signal_limit_is_the_linear_chain(mod)),
        ("nl_sat", lambda: pins.test_nonlinear_saturation_leaves_nothing_for_later_levels(mod)),
        ("nl_gelu", lambda: pins.test_nonlinear_chain_against_library_gelu(mod)),
    ]
    for name, fn in cases:
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found once: {name}"
    src = tmp_path / "mut.c"
    src.write_text(text.replace(old, new))
    lib = prism_oracle.build(force=True, src=str(src), lib_path=str(tmp_path / "libmut.so"))
    mod = prism_oracle.OracleLib(lib)
    failed = _pin_suite(mod)
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_the_suite(oracle_mod):
    assert _pin_suite(oracle_mod) == []
