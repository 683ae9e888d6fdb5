"""Each plausible mistake planted in a copy of the oracle must fail a pin.

The mistakes are planted on the CPU, in a temporary copy of the oracle's C
source; the committed oracle is never changed.  Every mutant keeps all memory
accesses in bounds.
"""
import functools
import os
import types

import pytest

import oracle
from tests import _pins

MUTANTS = {
    "decay_sign": ("alpha[i] = exp(gt[i]);", "alpha[i] = exp(-gt[i]);"),
    "decay_on_value_columns": ("S[i * dv + j] *= alpha[i];",
                               "S[i * dv + j] *= alpha[j % dk];"),
    "decay_dropped": ("S[i * dv + j] *= alpha[i];", "S[i * dv + j] *= 1.0;"),
    "error_sign": ("err[j] = vt[j] - pred;", "err[j] = vt[j] + pred;"),
    "no_delta_correction": ("err[j] = vt[j] - pred;", "err[j] = vt[j];"),
    "beta_dropped": ("const double bk = bt * kt[i];", "const double bk = kt[i];"),
    "readout_with_key": ("acc += S[i * dv + j] * qt[i];",
                         "acc += S[i * dv + j] * kt[i];"),
    "readout_before_write": ("acc += S[i * dv + j] * qt[i];",
                             "acc += (S[i * dv + j] - bt * kt[i] * err[j]) * qt[i];"),
    "prediction_undecayed": ("pred += S[i * dv + j] * kt[i];",
                             "pred += S[i * dv + j] * kt[i] / alpha[i];"),
    "prediction_with_query": ("pred += S[i * dv + j] * kt[i];",
                              "pred += S[i * dv + j] * qt[i];"),
    "beta_head_index": ("const double bt = J->beta[t * H + h];",
                        "const double bt = J->beta[t * H];"),
    "query_head_index": ("const double *qt = J->q + (t * H + h) * dk;",
                         "const double *qt = J->q + (t * H) * dk;"),
    "initial_state_unit": ("memcpy(S, J->S0 + state_off,", "memcpy(S, J->S0,"),
    "first_token_skipped": ("for (int64_t t = J->cu_seqlens[n]; t",
                            "for (int64_t t = J->cu_seqlens[n] + (n > 0); t"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation site must be unique: %r" % old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_library(str(path),
                                                     str(tmp_path / "libm.so")))
    handle = types.SimpleNamespace(
        prefill=functools.partial(oracle.prefill, lib=lib),
        decode_step=functools.partial(oracle.decode_step, lib=lib))
    failed = []
    for pin in _pins.PINS:
        try:
            pin(handle)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
