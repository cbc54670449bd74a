"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a textual edit of a copy of ``oracle/kda_oracle.c`` compiled to
a temporary library; the pin tests of ``test_oracle_pins`` are then run with
the mutant loaded in place of the real oracle. The real source is untouched.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTANTS = {
    "decay_rows_not_columns": ("S[(size_t)r * K + c] *= alpha[c];", "S[(size_t)r * K + c] *= alpha[r % K];"),
    "decay_dropped": ("S[(size_t)r * K + c] *= alpha[c];", "S[(size_t)r * K + c] *= 1.0;"),
    "delta_sign": ("double e = beta * (v[r] - pred[r]);", "double e = beta * (v[r] + pred[r]);"),
    "prediction_transposed": ("s += S[(size_t)r * K + c] * k[c];", "s += S[(size_t)c * K + r] * k[c];"),
    "output_unscaled": ("o[r] = scale * s;", "o[r] = s;"),
    "output_reads_key": ("s += S[(size_t)r * K + c] * q[c];", "s += S[(size_t)r * K + c] * k[c];"),
    "gate_sign": ("alpha[c] = exp(lower_bound * sigmoid(xg[c]));", "alpha[c] = exp(lower_bound * sigmoid(-xg[c]));"),
    "gate_no_sigmoid": ("alpha[c] = exp(lower_bound * sigmoid(xg[c]));", "alpha[c] = exp(lower_bound * xg[c]);"),
    "A_log_not_exponentiated": ("double a = A_log ? exp((double)A_log[h]) : 1.0;\n        for (int64_t t",
                                "double a = A_log ? (double)A_log[h] : 1.0;\n        for (int64_t t"),
    "bias_outside": ("xg[c] = a * (widen_bf16(g[rk + c]) + b);", "xg[c] = a * widen_bf16(g[rk + c]) + b;"),
    "beta_not_activated": ("double bt = sigmoid(widen_bf16(beta[(size_t)t * H + h]));",
                           "double bt = widen_bf16(beta[(size_t)t * H + h]);"),
    "varlen_state_slot": ("*slot = seq;", "*slot = 0;"),
    "qk_norm_skips_q": ("qq[c] *= fq;", "qq[c] *= 1.0;"),
    "qk_norm_no_sqrt": ("double fk = 1.0 / sqrt(sk + 1e-6), fq = 1.0 / sqrt(sq + 1e-6);",
                        "double fk = 1.0 / (sk + 1e-6), fq = 1.0 / (sq + 1e-6);"),
    "gate_entry_A_log": ("double a = A_log ? exp((double)A_log[h]) : 1.0;\n            for (int c",
                         "double a = A_log ? (double)A_log[h] : 1.0;\n            for (int c"),
}

PIN_TESTS = [
    pins.test_single_token_from_zero_state,
    pins.test_single_token_with_state_matrix_form,
    pins.test_beta_zero_is_pure_decay,
    pins.test_delta_rule_storage_orthonormal_keys,
    pins.test_delta_rule_storage_through_full_gate,
    pins.test_gate_special_points,
    lambda: pins.test_chunked_wy_agrees("b1_t64_h1", {}, 16),
    lambda: pins.test_chunked_wy_agrees("varlen_n16_h32", dict(lengths=[5, 37, 16, 1, 23], H=2), 16),
    pins.test_varlen_equals_separate_calls,
    pins.test_split_call_state_carry,
    pins.test_scale_is_linear_on_output_only,
    pins.test_qk_l2norm_invariant_to_power_of_two_input_scale,
    pins.test_qk_l2norm_delta_rule_storage_with_scaled_one_hot_keys,
]


def _build_mutant(tmpdir, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    path = os.path.join(tmpdir, name + ".c")
    with open(path, "w") as f:
        f.write(text.replace(old, new))
    so = os.path.join(tmpdir, name + ".so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", so, path, "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    old, new = MUTANTS[name]
    real = oracle._load()
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, name, old, new)
        lib = ctypes.CDLL(so)
        for fn in ("kda_oracle_fwd", "kda_oracle_core", "kda_oracle_gate"):
            getattr(lib, fn).argtypes = getattr(real, fn).argtypes
            getattr(lib, fn).restype = getattr(real, fn).restype
        monkeypatch.setattr(oracle, "_lib", lib)
        caught = []
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(getattr(t, "__name__", "chunked"))
        assert caught, f"mutant {name} passed every pin"
