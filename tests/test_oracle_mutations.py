"""The oracle's pins are sensitive: plant a plausible mistake in a copy of the
C oracle (on the CPU), rebuild it, and check that at least one pin fails.

Each mutation is a one-line textual change of ``oracle/kda_oracle.c``: a
dropped term, a wrong sign, a wrong operand or index, a transposed state.
"""
import ctypes
import os
import subprocess

import pytest

from oracle import recurrence
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(recurrence.__file__), "kda_oracle.c")

MUTATIONS = {
    "dropped decay": ("Sr[c] *= dec[c];", "Sr[c] *= 1.0;"),
    "decay on value rows": ("Sr[c] *= dec[c];", "Sr[c] *= dec[r % K];"),
    "prediction uses q": ("pred += Sr[c] * kt[c];", "pred += Sr[c] * qt[c];"),
    "wrong delta sign": ("double w = b * ((double)vr[r] - pred);",
                         "double w = b * ((double)vr[r] + pred);"),
    "write uses q": ("Sr[c] += w * kt[c];", "Sr[c] += w * qt[c];"),
    "read-out uses k": ("o += Sr[c] * qt[c];", "o += Sr[c] * kt[c];"),
    "softplus sign": (": -amul * oracle_softplus(z);", ": -amul * oracle_softplus(-z);"),
    "dropped A_log multiplier": ("lower_bound * oracle_sigmoid(amul * z)",
                                 "lower_bound * oracle_sigmoid(z)"),
    "dropped dt_bias": ("(dt_bias ? (double)dt_bias[h * K + c] : 0.0)", "0.0"),
    "beta without sigmoid": (": oracle_sigmoid((double)beta[t * H + h]);",
                             ": (double)beta[t * H + h];"),
    "beta-as-probability mode still applies the sigmoid": (
        "double b = beta_is_prob ? (double)beta[t * H + h] :",
        "double b = beta_is_prob ? oracle_sigmoid((double)beta[t * H + h]) :"),
    "log-space gate takes the bias": ("double a = (gate_mode == ORACLE_GATE_LOGSPACE) ? (double)gr[c]",
                                      "double a = (gate_mode == ORACLE_GATE_LOGSPACE) ? z"),
    "transposed initial state": ("init[(n * H + h) * V * K + i]",
                                 "init[(n * H + h) * V * K + (i % K) * V + i / K]"),
    "l2 norm without sqrt": ("double rq = 1.0 / sqrt(nq + l2_eps)",
                             "double rq = 1.0 / (nq + l2_eps)"),
    "scale dropped": ("out[(t * H + h) * V + r] = scale * o;", "out[(t * H + h) * V + r] = o;"),
}


def _pin_suite():
    """Run the core pins; return the names of those that fail."""
    failed = []
    checks = [
        ("exact rational safe", lambda: pins.test_exact_rational_example("safe")),
        ("exact rational unsafe", lambda: pins.test_exact_rational_example("unsafe")),
        ("affine safe", lambda: pins.test_affine_map_brute_force(3, 2, 4, "safe")),
        ("affine unsafe", lambda: pins.test_affine_map_brute_force(2, 3, 4, "unsafe")),
        ("affine logspace, beta given", lambda: pins.test_affine_map_brute_force_modes(3, 2, 4)),
        ("beta zero", lambda: pins.test_beta_zero_closed_form("unsafe")),
        ("gate", pins.test_gate_through_c_recurrence),
        ("fixed point", pins.test_delta_rule_fixed_point),
        ("l2 invariance", pins.test_l2norm_scale_invariance),
    ]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_suite():
    assert _pin_suite() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                           str(mutated), "-lm"])
    lib = recurrence.configure(ctypes.CDLL(str(so)))
    monkeypatch.setattr(recurrence, "_lib", lib)
    failed = _pin_suite()
    assert failed, f"planted mistake '{name}' passed every pin"
