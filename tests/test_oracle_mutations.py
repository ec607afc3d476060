"""Each reading slip the entmax oracle could carry is caught by a committed pin: the slip is
planted in a copy of oracle/entmax.py (on the CPU, by a source substitution; the oracle file
itself is untouched), and at least one pin of test_oracle_entmax.py must then fail."""

import importlib.util
import os
import sys

import pytest

import oracle
import test_oracle_entmax as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "entmax.py")

# (name, the oracle's text, the slip)
SLIPS = [
    ("divisor 12 -> 4", "((hi - lo) ** 2 / 12.0)", "((hi - lo) ** 2 / 4.0)"),
    ("q_d^2 -> |q_d|", "@ (qh * qh)", "@ np.abs(qh)"),
    ("(scale/2) unsquared", "v_b[h] = half * half *", "v_b[h] = half *"),
    ("page-weighted mu and sigma^2",
     "        mu = (n_tok * c[h]).sum() / N\n"
     "        var = (n_tok * (c[h] - mu) ** 2).sum() / N + (n_tok * v[h]).sum() / N\n",
     "        mu = c[h].mean()\n"
     "        var = ((c[h] - mu) ** 2).mean() + v[h].mean()\n"),
]


def mutated_module(old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"the oracle no longer holds {old!r}"
    name = "oracle._entmax_slip"
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    sys.modules[name] = mod
    try:
        exec(compile(text.replace(old, new), SRC + " (planted slip)", "exec"), mod.__dict__)
    finally:
        del sys.modules[name]
    return mod


def pins_fail(E):
    checks = [lambda: pins.check_page_moments_golden(E),
              lambda: [pins.check_page_moments_monte_carlo(E, s) for s in (0, 1, 2)],
              lambda: pins.check_select_golden(E),
              lambda: pins.check_token_weighting(E)]
    failed = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            failed += 1
    return failed


def test_the_unmutated_oracle_passes_every_pin():
    assert pins_fail(mutated_module("import math", "import math")) == 0


@pytest.mark.parametrize("name,old,new", SLIPS, ids=[s[0] for s in SLIPS])
def test_every_planted_slip_fails_a_pin(name, old, new):
    assert pins_fail(mutated_module(old, new)) >= 1, name
