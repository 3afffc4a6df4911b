"""The projection oracle's pins are sensitive: plant one plausible mistake at a time in a copy of
oracle/prism_projection.py (on the CPU), load it, and check that at least one pin fails."""
import importlib.util
import os

import pytest

import tests.test_projection_oracle as pins
from oracle import prism_projection

SRC = prism_projection.__file__

MUTATIONS = [
    ("taps reversed", "a[:, j:, :] += w[j][None, None, :] * X[:, : T - j, :]",
     "a[:, j:, :] += w[3 - j][None, None, :] * X[:, : T - j, :]"),
    ("anchor looks ahead", "a[:, j:, :] += w[j][None, None, :] * X[:, : T - j, :]",
     "a[:, : T - j, :] += w[j][None, None, :] * X[:, j:, :]"),
    ("basis not normalised", "u = np.where(norm > 0, yu / np.where(norm > 0, norm, 1.0), 0.0)", "u = yu"),
    ("head and level swapped", "yu = Y[..., :NU].reshape(B, T, H, R, dk).transpose(0, 2, 1, 3, 4)",
     "yu = Y[..., :NU].reshape(B, T, R, H, dk).transpose(0, 3, 1, 2, 4)"),
    ("gain block offset", "p = Y[..., NU:NU + NP]", "p = Y[..., NU - 1:NU + NP - 1]"),
    ("gate without logistic", "gamma = 1.0 / (1.0 + np.exp(-g))", "gamma = g"),
    ("weights transposed in the product", "Y = a @ W.T  # [B, T, N]", "Y = (a @ W.T)[..., ::-1]  # [B, T, N]"),
]


def _load(path):
    spec = importlib.util.spec_from_file_location("mutated_projection", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pin_suite(mod):
    failed = []
    saved = pins.PP
    pins.PP = mod
    try:
        for name in ("test_anchor_is_numpy_causal_convolution", "test_basis_is_unit_and_scale_invariant",
                     "test_gain_is_linear_and_gate_is_a_logistic", "test_weight_layout_by_one_hot_rows",
                     "test_batches_do_not_leak_through_the_convolution"):
            try:
                getattr(pins, name)()
            except (AssertionError, ValueError, IndexError):
                failed.append(name)
    finally:
        pins.PP = saved
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found once: {name}"
    path = os.path.join(tmp_path, "mut.py")
    with open(path, "w") as f:
        f.write(text.replace(old, new))
    assert _pin_suite(_load(path)), f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_the_suite():
    assert _pin_suite(prism_projection) == []
