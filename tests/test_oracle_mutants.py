"""Each planted mistake in a copy of the oracle must fail at least one pin.

The mistakes are the plausible ones: a transposed mixture weight, a dropped
term, a wrong sign, a swapped operand, the wrong reduction in a gradient, a
missing max subtraction, a swapped endpoint branch. The copy is compiled into
a temporary directory on the CPU; the committed oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle_pins
from oracle import oracle as O

MUTANTS = {
    "mixture weights transposed": ("const real lw_s = RLOG(1.0 - beta);", "const real lw_s = RLOG(beta);"),
    "dropped (1-beta) in the loss": ("real value = beta * a + (1.0 - beta) * b;", "real value = beta * a + b;"),
    "wrong sign of B in dS": ("(lp - lm - b)", "(lp - lm + b)"),
    "A used in place of B in dS": ("(lp - lm - b)", "(lp - lm - a)"),
    "operands swapped in KL": ("csum_add(&kl, REXP(la) * (la - lb));", "csum_add(&kl, REXP(la) * (lb - la));"),
    "forward/reverse branches swapped": ("return kl_row(V, t, s, g, dt, ds);", "return kl_row(V, s, t, g, ds, dt);"),
    "entropy gradient sign": ("(lp + value)", "(lp - value)"),
    "log-prob gradient sign": ("dxr[j] -= REXP(log_prob(&st, xr[j])) * gs;", "dxr[j] += REXP(log_prob(&st, xr[j])) * gs;"),
    "max not subtracted": ("csum_add(&z, REXP(v - r.m));", "csum_add(&z, REXP(v));"),
    "min instead of max": ("if (v > r.m)", "if (v < r.m && r.m != -INFINITY || r.m == -INFINITY)"),
    "KL gradient target index": ("db[j] = g * (b - a);", "db[j] = g * (a - b);"),
    "teacher weight in dT": ("g * beta * REXP(lq)", "g * (1.0 - beta) * REXP(lq)"),
    "support violation ignored": ("if (xa[j] != -INFINITY && xb[j] == -INFINITY) {",
                                  "if (0 && xa[j] != -INFINITY && xb[j] == -INFINITY) {"),
    "empty segment not skipped": ("if (!r.empty)\n            csum_add(&z, r.z * REXP(r.m - m));",
                                  "csum_add(&z, r.z * REXP(r.m - m));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    with open(O.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{name}' must be unique"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.run(O.compile_command(str(mutant_c), lib_path), check=True)
    monkeypatch.setattr(O, "_lib", O.load(lib_path))
    failed = []
    for pin in oracle_pins.PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"


# Planted mistakes in the Python compositions of the oracle (fused-linear JSD,
# cross-entropy, teacher top-k forward KL): the function is re-created from its
# own source with one edit and swapped in for the duration of the test.
PY_MUTANTS = {
    "linear: teacher gradient used for the student head": ("jsd_linear", "ds.T @ h_s", "dt.T @ h_s"),
    "linear: student head used for the teacher logits": ("jsd_linear", "t = h_t @ w_t.T", "t = h_t @ w_t.T + s * 0.01"),
    "cross-entropy: temperature multiplies the gradient": ("cross_entropy", "dx = dx / float(temperature)",
                                                            "dx = dx * float(temperature)"),
    "cross-entropy: sign": ("cross_entropy", "loss = -out[:, 0]", "loss = out[:, 0]"),
    "top-k KL: log-probs used as weights": ("topk_forward_kl", "np.exp(np.where(live, tl, 0.0))",
                                            "np.where(live, tl, 0.0)"),
    "top-k KL: temperature ignored": ("topk_forward_kl", "logprobs(s / float(temperature)", "logprobs(s"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_composition_mistake_is_caught(name, monkeypatch):
    import inspect
    import textwrap

    fn_name, old, new = PY_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(O, fn_name)))
    assert src.count(old) == 1, f"mutation site for '{name}' must be unique"
    namespace = dict(vars(O))
    exec(compile(src.replace(old, new), f"<mutant {fn_name}>", "exec"), namespace)
    monkeypatch.setattr(O, fn_name, namespace[fn_name])
    failed = []
    for pin in oracle_pins.PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
