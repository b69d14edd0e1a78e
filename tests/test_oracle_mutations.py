"""The pins must catch a plausible mistake in the oracle.

Each case copies oracle.c to a temporary directory, plants one mistake (a
dropped term, a wrong sign, a wrong index, a swapped operand), builds it, and
checks that at least one pin fails against the mutant.  Nothing here touches the
real oracle or any GPU.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle.oracle as orc_mod
from oracle import Problem

SRC = os.path.join(os.path.dirname(orc_mod.__file__), "oracle.c")

MUTATIONS = [
    ("drop_log1p_in_softplus", "if (x > 0.0) return x + log1p(exp(-x));", "if (x > 0.0) return x;"),
    ("target_included_in_sum", "if (j != skip) s += exp(x[j] - m);", "s += exp(x[j] - m);"),
    ("wrong_sign_target_grad", "? -exp(s.lse_nt - s.lse) : p;", "? exp(s.lse_nt - s.lse) : p;"),
    ("z_grad_missing_factor_2", "double term = w_ce * p_minus_onehot + 2.0 * alpha * s.lse * p;",
     "double term = w_ce * p_minus_onehot + alpha * s.lse * p;"),
    ("kl_operands_swapped", "term += w_kl * (p_tau - q) / temperature;", "term += w_kl * (q - p_tau) / temperature;"),
    ("kl_wrong_log_term", "kl += q * (log_q - (b[j] - lse_b));", "kl += q * (log_q - (b[j] - lse_a));"),
    ("logaddexp_wrong_sign", "return hi + log1p(exp(lo - hi));", "return hi - log1p(exp(lo - hi));"),
    ("gspo_coef_uses_onehot_only", "g[j] = s_tok * term + c_r * p_minus_onehot;", "g[j] = s_tok * term + c_r * p;"),
    ("entropy_drops_log1p_for_others", "double nlogp = (j == k) ? l1 : (z[k] - z[j]) + l1;",
     "double nlogp = (j == k) ? l1 : (z[k] - z[j]);"),
    ("entropy_max_term_rounds_to_zero", "double nlogp = (j == k) ? l1 :", "double nlogp = (j == k) ? 0.0 :"),
    ("wrong_row_stride", "out[j] = orc_elem(dtype, base, r * ld + j);", "out[j] = orc_elem(dtype, base, r * V + j);"),
    ("bf16_decode_wrong_shift", "[idx] << 16;", "[idx] << 15;"),
    ("kl_grad_times_tau", "term += w_kl * (p_tau - q) / temperature;", "term += w_kl * (p_tau - q) * temperature;"),
    ("teacher_not_tempered", "a[j] = u[j] / tau;", "a[j] = u[j];"),
]


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    real = orc_mod._load()
    lib.orc_forward.argtypes = real.orc_forward.argtypes
    lib.orc_forward.restype = ctypes.c_int
    lib.orc_grad.argtypes = real.orc_grad.argtypes
    lib.orc_grad.restype = ctypes.c_int
    lib.orc_entropy.argtypes = real.orc_entropy.argtypes
    lib.orc_entropy.restype = ctypes.c_int
    return lib


def _pins_pass():
    """A compact set of the pins; returns False as soon as one fails."""
    import tests.test_oracle_pins as pins
    from tests.conftest import read_golden
    checks = [
        lambda: pins.test_worked_example_margin20(read_golden, 1000),
        lambda: pins.test_worked_example_v2_exact(),
        lambda: pins.test_uniform_logits(7, -3.5),
        lambda: pins.test_two_class_closed_form(1),
        lambda: pins.test_row_sums(),
        lambda: pins.test_torch_fp64_autograd(0),
        lambda: pins.test_gspo_ratio_one(),
        lambda: pins.test_entropy_uniform_is_log_v(9),
        lambda: pins.test_entropy_two_class_and_brute(),
        lambda: pins.test_entropy_confident_rows(60.0),
        lambda: pins.test_brute_force_mpmath("kl_tau2", 2, 3, dict(teacher=True, kl_weight=0.7,
                                                                    temperature=2.0, z_alpha=0.01)),
        lambda: pins.test_bf16_inputs_match_fp32_bit_for_bit(),
        lambda: pins.test_two_class_closed_form_temperature(0.5),
        lambda: pins.test_torch_fp64_autograd_temperature(3.0),
        lambda: pins.test_kl_shift_invariance(0.25),
    ]
    # the stride mutation only shows with ld > V
    z = np.random.default_rng(0).normal(size=(3, 8)).astype(np.float32)
    wide = np.zeros((3, 11), dtype=np.float32)
    wide[:, :8] = z
    t = np.array([1, 2, 3])
    def stride_check():
        a = oracle.forward(Problem(logits=z, V=8, targets=t)).total
        b = oracle.forward(Problem(logits=wide, V=8, targets=t)).total
        assert a == b
    checks.append(stride_check)
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


def test_real_oracle_passes_compact_pins():
    assert _pins_pass()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, name, old, new, monkeypatch):
    lib = _build_mutant(tmp_path, old, new)
    monkeypatch.setattr(orc_mod, "_lib", lib)
    assert not _pins_pass(), f"mutation {name} survived the pins"
