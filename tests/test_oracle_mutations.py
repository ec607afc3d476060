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
    ("2-entmax weights (no square)", "p = np.maximum(z - tau, 0.0) ** 2",
     "p = np.maximum(z - tau, 0.0)"),
    ("support not checked against its root", "support = np.nonzero(ok & (tau_k < zs))[0]",
     "support = np.nonzero(ok)[0]"),
    ("z = x, not x / 2, in the attention", "p, t = entmax15(x / 2.0)", "p, t = entmax15(x)"),
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
              lambda: pins.check_token_weighting(E),
              lambda: pins.check_entmax15(E),
              lambda: pins.check_entmax_attend_golden(E)]
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


# ---- the attention oracle (oracle/kvattn.py) against test_oracle_pins.py -----------------

import inspect

import test_oracle_pins as attn_pins

KV_SRC = os.path.join(os.path.dirname(oracle.__file__), "kvattn.py")

KV_SLIPS = [
    ("mean in place of the minimum", "mn[P] = keys.min(axis=1)", "mn[P] = keys.mean(axis=1)"),
    ("the min side of the bound dropped",
     "total += np.maximum(qh * lo, qh * hi).sum(axis=1)", "total += (qh * hi).sum(axis=1)"),
    ("ties to the higher page index", "order = np.lexsort((np.arange(n), -s))",
     "order = np.lexsort((-np.arange(n), -s))"),
    ("keep count rounded down", "return min(n, max(1, math.ceil(ratio * n - 1e-9)))",
     "return min(n, max(1, int(ratio * n)))"),
    ("softmax scale dropped", "x = scale * (K @ qh)", "x = K @ qh"),
    ("lse without the max", "lse[b, h] = M + np.log(L)", "lse[b, h] = np.log(L)"),
    ("merge weights with the wrong sign", "w = np.exp(m[live] - M)", "w = np.exp(M - m[live])"),
    ("dropped mass of the kept tokens", "delta[b, h] = w[~tok_keep].sum() / w.sum()",
     "delta[b, h] = w[tok_keep].sum() / w.sum()"),
    ("last page one token long",
     "return max(0, min(int(page_size), int(seq_len) - int(p) * int(page_size)))",
     "return max(0, min(int(page_size), int(seq_len) - int(p) * int(page_size) + 1))"),
    ("page count rounded down", "return -(-int(seq_len) // int(page_size))",
     "return int(seq_len) // int(page_size)"),
    ("local window one page too long", "forced[max(0, n - int(local)):] = True",
     "forced[max(0, n - int(local) - 1):] = True"),
]


def pin_calls(pins):
    """Every pin of a pin module callable with its first parametrisation."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        kwargs = {}
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = mark.args[0]
            names = [a.strip() for a in names.split(",")] if isinstance(names, str) else list(names)
            first = mark.args[1][0]
            kwargs.update({names[0]: first} if len(names) == 1 else dict(zip(names, first)))
        if set(inspect.signature(fn).parameters) <= set(kwargs):
            calls.append((name, fn, kwargs))
    return calls


def attn_pins_fail(monkeypatch, old, new):
    text = open(KV_SRC).read()
    assert text.count(old) == 1, f"the oracle no longer holds {old!r}"
    name = "oracle._kvattn_slip"
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(text.replace(old, new), KV_SRC + " (planted slip)", "exec"), mod.__dict__)
    for attr, val in vars(mod).items():
        if inspect.isfunction(val) and val.__module__ == name:
            for target in (oracle, oracle.kvattn):
                if hasattr(target, attr):
                    monkeypatch.setattr(target, attr, val)
    failed = []
    for pin, fn, kwargs in pin_calls(attn_pins):
        try:
            fn(**kwargs)
        except Exception:                       # an assertion, or a crash on bad shapes
            failed.append(pin)
    return failed


def test_the_unmutated_attention_oracle_passes_every_pin(monkeypatch):
    assert len(pin_calls(attn_pins)) >= 20
    assert attn_pins_fail(monkeypatch, "import math", "import math") == []


@pytest.mark.parametrize("name,old,new", KV_SLIPS, ids=[s[0] for s in KV_SLIPS])
def test_every_planted_attention_slip_fails_a_pin(monkeypatch, name, old, new):
    assert attn_pins_fail(monkeypatch, old, new), name


# ---- the FP8 statistics oracle (oracle/fp8stats.py) against test_oracle_fp8.py -----------

import test_oracle_fp8 as fp8_pins

FP8_SRC = os.path.join(os.path.dirname(oracle.__file__), "fp8stats.py")

FP8_SLIPS = [
    ("the minimum rounded up", "code_mn[rows] = quantize_down(lo, e[:, :, None])",
     "code_mn[rows] = quantize_up(lo, e[:, :, None])"),
    ("row exponent one too large", "e = np.maximum(e, MIN_EXPONENT)",
     "e = np.maximum(e, MIN_EXPONENT) + 1"),
    ("subnormal scale 2^-7", "return sign * (mant / 8.0) * 2.0 ** -6",
     "return sign * (mant / 8.0) * 2.0 ** -7"),
    ("an on-grid value rounded down a step", 'idx = np.searchsorted(vals, a, side="right") - 1',
     'idx = np.searchsorted(vals, a, side="left") - 1'),
]


def fp8_pins_fail(monkeypatch, old, new):
    text = open(FP8_SRC).read()
    assert text.count(old) == 1, f"the oracle no longer holds {old!r}"
    name = "oracle._fp8stats_slip"
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(text.replace(old, new), FP8_SRC + " (planted slip)", "exec"), mod.__dict__)
    for attr, val in vars(mod).items():
        if inspect.isfunction(val) and val.__module__ == name:
            for target in (oracle, oracle.fp8stats):
                if hasattr(target, attr):
                    monkeypatch.setattr(target, attr, val)
            if hasattr(fp8_pins, attr):
                monkeypatch.setattr(fp8_pins, attr, val)
    failed = []
    for pin, fn, kwargs in pin_calls(fp8_pins):
        try:
            fn(**kwargs)
        except Exception:
            failed.append(pin)
    return failed


def test_the_unmutated_fp8_oracle_passes_every_pin(monkeypatch):
    assert len(pin_calls(fp8_pins)) >= 5
    assert fp8_pins_fail(monkeypatch, "import numpy as np", "import numpy as np") == []


@pytest.mark.parametrize("name,old,new", FP8_SLIPS, ids=[s[0] for s in FP8_SLIPS])
def test_every_planted_fp8_slip_fails_a_pin(monkeypatch, name, old, new):
    assert fp8_pins_fail(monkeypatch, old, new), name
