"""Each plausible mistake planted in a copy of the oracle's gate prologue must
fail one of its pins ("[논문 리뷰] Kimi K3 Technical Report", section 3.5:
g = g_min Sigmoid(e^A z) with g_min = -5).

The mistakes are planted in a private copy of the function's source, compiled
into a throw-away module; the committed oracle is never changed.
"""
import inspect
import textwrap
import types

import numpy as np
import pytest

import oracle
from tests import test_oracle_prologue as pins

MUTANTS = {
    "exp_of_minus_A": ("np.exp(A) * z", "np.exp(-A) * z"),
    "no_exp_on_A": ("np.exp(A) * z", "A * z"),
    "A_added": ("np.exp(A) * z", "np.exp(A) + z"),
    "sigmoid_sign": ("np.tanh(0.5 * s)", "np.tanh(-0.5 * s)"),
    "sigmoid_scale": ("np.tanh(0.5 * s)", "np.tanh(s)"),
    "g_min_positive": ("g = G_MIN * 0.5", "g = -G_MIN * 0.5"),
    "q_scale_dropped": ("float(q_scale) / qn", "1.0 / qn"),
    "k_not_normalised": ("k / kn", "k"),
}


def _mutant_module(old, new):
    src = textwrap.dedent(inspect.getsource(oracle.gate_prologue))
    assert src.count(old) == 1, "mutation site must be unique: %r" % old
    mod = types.ModuleType("gate_mutant")
    mod.np = np
    mod.G_MIN = oracle.G_MIN
    mod._c64 = oracle._c64
    exec(compile(src.replace(old, new), "<gate_mutant>", "exec"), mod.__dict__)
    shim = types.SimpleNamespace(gate_prologue=mod.gate_prologue, G_MIN=oracle.G_MIN)
    return shim


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_gate_mutant_is_caught(name, monkeypatch):
    old, new = MUTANTS[name]
    shim = _mutant_module(old, new)
    monkeypatch.setattr(pins, "oracle", shim)
    failed = []
    for pin in (pins.test_gate_values_and_bounds, pins.test_qk_normalisation,
                pins.test_gate_value_with_nonzero_A):
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every gate pin" % name


def test_exp_minus_A_fails_the_nonzero_A_pin(monkeypatch):
    # The slip the other pins cannot see: only the value pin at A != 0 fails.
    monkeypatch.setattr(pins, "oracle", _mutant_module(*MUTANTS["exp_of_minus_A"]))
    pins.test_gate_values_and_bounds()
    pins.test_qk_normalisation()
    with pytest.raises(AssertionError):
        pins.test_gate_value_with_nonzero_A()
