"""The backward oracle's pins are sensitive: plant one plausible mistake at a time in a copy
of its source (on the CPU), rebuild it, and check that the finite-difference pins fail."""
import numpy as np
import pytest

import tests.test_backward_oracle as pins
from oracle import prism_backward, prism_oracle

SRC = prism_backward._SRC

# (name, text in the backward source, replacement)
MUTATIONS = [
    ("state carry without decay", "dS[(size_t)i * dk + j] = al * (dS[(size_t)i * dk + j] - be * z[i] * kt[j]);",
     "dS[(size_t)i * dk + j] = (dS[(size_t)i * dk + j] - be * z[i] * kt[j]);"),
    ("state carry sign", "dS[(size_t)i * dk + j] = al * (dS[(size_t)i * dk + j] - be * z[i] * kt[j]);",
     "dS[(size_t)i * dk + j] = al * (dS[(size_t)i * dk + j] + be * z[i] * kt[j]);"),
    ("readout term dropped", "dS[(size_t)i * dk + j] += dOt[i] * qt[j];", "dS[(size_t)i * dk + j] += 0.0;"),
    ("readout term transposed", "dS[(size_t)i * dk + j] += dOt[i] * qt[j];",
     "dS[(size_t)i * dk + j] += dOt[j % dv] * qt[i % dk];"),
    ("dq from the pre-update state", "const double *St = t + 1 < T ? Sprev + (size_t)(t + 1) * DD : S;",
     "const double *St = P;"),
    ("dbeta without the delta term", "dbeta[t] = vz - al * yz;", "dbeta[t] = vz;"),
    ("dalpha without the delta term", "dalpha[t] = dSP - be * yz;", "dalpha[t] = dSP;"),
    ("dk without the state term", "- al * be * P[(size_t)i * dk + j] * z[i];", ";"),
    ("dk with the key in place of v", "(be * vt[i] - al * be * y[i])", "(be * kt[i % dk] - al * be * y[i])"),
    ("write cotangent dropped", "dvv[(size_t)t * dv + i] += be * z[i];", "dvv[(size_t)t * dv + i] += 0.0;"),
    ("du along the wrong axis", "s += dS[(size_t)i * dk + j] * xt[(size_t)l * dv + i];",
     "s += dS[(size_t)j % dv * dk + i % dk] * xt[(size_t)l * dv + i];"),
    ("chain carry sign", "dr_next = gm * g * dxl + (1.0 - et * g) * dr_next;",
     "dr_next = gm * g * dxl + (1.0 + et * g) * dr_next;"),
    ("gain cotangent without the chain term", "dg += gm * rl * dxl - et * rl * dr_next;", "dg += gm * rl * dxl;"),
    ("deta sign", "deta[(size_t)t * R + l] += -g * rl * dr_next;", "deta[(size_t)t * R + l] += g * rl * dr_next;"),
    ("gain derivative without the h^2 term", "ph * (2.0 - hc * hc) * dg", "ph * 2.0 * dg"),
    ("residual derivative with Phi only", "dh[(size_t)t * dv + c] = -g * dr_next + ph",
     "dh[(size_t)t * dv + c] = -Ph * dr_next + ph"),
    ("non-linear step cotangent sign", "const double ddelta = gm * dxl - dr_next;",
     "const double ddelta = gm * dxl + dr_next;"),
    ("non-linear gain cotangent from the gain", "dpg[((size_t)t * R + l) * dv + c] = dz * rl;",
     "dpg[((size_t)t * R + l) * dv + c] = dz * p;"),
    ("non-linear GELU derivative without z phi", "const double dz = ddelta * (Phi_of(zz) + zz * phi_of(zz));",
     "const double dz = ddelta * Phi_of(zz);"),
    ("non-linear residual derivative dropped", "dh[(size_t)t * dv + c] = -g * dr_next;  /*",
     "dh[(size_t)t * dv + c] = 0.0 * dr_next;  /*"),
    ("conv transpose taps reversed", "dvv[(size_t)src * dv + c] += w[j * dv + c] * d;",
     "dvv[(size_t)src * dv + c] += w[(3 - j) * dv + c] * d;"),
    ("conv weight cotangent from the wrong token", "dw[j * dv + c] += v[(size_t)src * dv + c] * d;",
     "dw[j * dv + c] += v[(size_t)t * dv + c] * d;"),
    ("history cotangent in reverse order", "a->dv_hist[(bh * 3 + (size_t)(3 + src)) * dv + c]",
     "a->dv_hist[(bh * 3 + (size_t)(-1 - src)) * dv + c]"),
    ("initial state ignored", "    if (a->S_init) memcpy(S,", "    if (0) memcpy(S,"),
]


def _pins_fail(mod):
    """Directional pins at L = 2 and 3 (linear chain) and L = 3 (non-linear chain) on the
    mutated build; True if any fails."""
    for L, nonlinear in ((2, False), (3, False), (3, True)):
        x, cot, L = pins.f64_case(L=L, T=13, nonlinear=nonlinear)
        try:
            g = pins.grads(x, cot, L, mod=mod)
        except (ValueError, OSError):
            return True
        for name in pins.inputs_of(x):
            err, _, _ = pins.directional_check(x, cot, L, name, g)
            if not np.isfinite(err) or err > 1e-8:
                return True
    return False


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found once: {name}"
    src = tmp_path / "mut.c"
    src.write_text(text.replace(old, new))
    lib = prism_oracle.build(force=True, src=str(src), lib_path=str(tmp_path / "libmut.so"))
    assert _pins_fail(prism_backward.BackwardLib(lib)), f"no pin caught the planted mistake '{name}'"


def test_unmutated_backward_passes():
    assert not _pins_fail(prism_backward)
