"""Every planted mistake in the oracle's sampled verify must be caught by a
pin (no GPU).

Each mutant is a copy of ``sampled_column``, ``sampled_decision`` and
``sampled_verify`` (their source text, from ``oracle/__init__.py``) with one
plausible error planted by text substitution, executed into a namespace of
its own; the test passes only when at least one pin of
``tests/pins_sampled.py`` rejects it.  The oracle itself is never modified.
"""
import inspect
import types

import numpy as np
import pytest

import oracle
from tests import pins_sampled

FUNCS = ("sampled_column", "sampled_decision", "sampled_verify")

MUTANTS = {
    "temperature_multiplies": [("z = [float(xi) / temperature", "z = [float(xi) * temperature")],
    "no_temperature": [("z = [float(xi) / temperature", "z = [float(xi) / 1.0")],
    "nucleus_strictly_above_top_p": [("if c >= top_p:", "if c > top_p:")],
    "nucleus_one_token_short": [("kept = [int(i) for i in ids[:last + 1]]", "kept = [int(i) for i in ids[:max(last, 1)]]"),
                                ("q = [p[t] / c for t in range(last + 1)]", "q = [p[t] / c for t in range(max(last, 1))]")],
    "nucleus_not_renormalised": [("q = [p[t] / c for t in range(last + 1)]", "q = [p[t] for t in range(last + 1)]")],
    "no_nucleus_cut": [("if c >= top_p:", "if False:")],
    "accept_at_equality": [("if u < qd:", "if u <= qd:")],
    "accept_compares_wrong_uniform": [("if u < qd:", "if u2 < qd:")],
    "draw_at_equality": [("if pick is None and run > target:", "if pick is None and run >= target:")],
    "residual_keeps_draft": [("        if draft is not None and tok == draft:\n            continue\n", ""),
                             ("if draft is None or tok != draft:\n            W += q[t]", "W += q[t]")],
    "residual_weight_not_rescaled": [("target = u2 * W", "target = u2")],
    "bonus_column_off_by_one": [("kept, q = sampled_column(vals[ln * (gamma + 1) + j]",
                                 "kept, q = sampled_column(vals[ln * (gamma + 1) + min(j, gamma - 1)]"),
                                ("ids[ln * (gamma + 1) + j], temperature",
                                 "ids[ln * (gamma + 1) + min(j, gamma - 1)], temperature")],
    "rejection_commits_draft": [("com[ln, j] = tok", "com[ln, j] = tok if ok or draft is None else draft")],
    "accept_length_counts_rejection": [("a = j\n", "a = j + 1 if j < gamma else j\n")],
    "top_k_ignored": [("vals, ids = topk(t, top_k, threads=threads)",
                       "vals, ids = topk(t, min(64, t.shape[1]), threads=threads)")],
    "shared_uniform_across_positions": [("float(u[ln, j, 0]), float(u[ln, j, 1])",
                                         "float(u[ln, 0, 0]), float(u[ln, 0, 1])")],
}


def _mutant(name):
    ns = {"np": np, "topk": oracle.topk}
    for f in FUNCS:
        src = inspect.getsource(getattr(oracle, f))
        for old, new in MUTANTS[name]:
            src = src.replace(old, new)
        exec(compile(src, f"<mutant {name}: {f}>", "exec"), ns)
    return types.SimpleNamespace(**{f: ns[f] for f in FUNCS})


def test_every_substitution_applies():
    srcs = "".join(inspect.getsource(getattr(oracle, f)) for f in FUNCS)
    for name, subs in MUTANTS.items():
        for old, _ in subs:
            assert old in srcs, f"mutant {name}: pattern not found: {old!r}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    oracle.load()
    impl = _mutant(name)
    caught = []
    for pin in pins_sampled.ALL_PINS:
        try:
            pin(impl)
        except (AssertionError, IndexError, KeyError, ValueError, TypeError, ZeroDivisionError, NameError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name!r}"
