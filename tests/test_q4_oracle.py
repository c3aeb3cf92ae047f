"""The Q4 shortlist head oracle against its pins, and planted mistakes in
copies of it that the pins must catch (no GPU).  See tests/pins_q4.py."""
import inspect
import types

import numpy as np
import pytest

import oracle
from oracle import q4head
from tests import pins_q4


@pytest.mark.parametrize("pin", pins_q4.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(q4head)


MUTANTS = {
    "nibbles_swapped": [("out[:, 0::2] = (b & 0x0F)", "out[:, 1::2] = (b & 0x0F)"),
                        ("out[:, 1::2] = (b >> 4)", "out[:, 0::2] = (b >> 4)")],
    "no_offset": [("(b & 0x0F).astype(np.int8) - 8", "(b & 0x0F).astype(np.int8)"),
                  ("(b >> 4).astype(np.int8) - 8", "(b >> 4).astype(np.int8)")],
    "offset_seven": [("(b & 0x0F).astype(np.int8) - 8", "(b & 0x0F).astype(np.int8) - 7"),
                     ("(b >> 4).astype(np.int8) - 8", "(b >> 4).astype(np.int8) - 7")],
    "signed_nibbles": [("(b & 0x0F).astype(np.int8) - 8", "(((b & 0x0F).astype(np.int8) ^ 8) - 8)"),
                       ("(b >> 4).astype(np.int8) - 8", "((((b >> 4)).astype(np.int8) ^ 8) - 8)")],
    "scale_of_next_block": [("return q * np.repeat(s, BLOCK, axis=1)", "return q * np.repeat(np.roll(s, -1, axis=1), BLOCK, axis=1)")],
    "one_scale_per_row": [("return q * np.repeat(s, BLOCK, axis=1)", "return q * s[:, :1]")],
    "rounded_through_float32": [("x = np.asarray(x, dtype=np.float64)", "x = np.asarray(x, dtype=np.float32).astype(np.float64)")],
    "truncated": [("r = np.rint(np.ldexp(x, 8 - e))", "r = np.trunc(np.ldexp(x, 8 - e))")],
    "ties_away_from_zero": [("r = np.rint(np.ldexp(x, 8 - e))", "r = np.sign(x) * np.floor(np.abs(np.ldexp(x, 8 - e)) + 0.5)")],
    "hidden_reversed": [("h = bf16_values(hidden)\n    if h.ndim == 1:\n        h = h[None, :]\n    rows = wq.shape[0]\n    out = np.empty((h.shape[0], rows), dtype=np.float64)\n    for r0 in range(0, rows, rows_per_block):\n        w = dequant(",
                         "h = bf16_values(hidden)[..., ::-1]\n    if h.ndim == 1:\n        h = h[None, :]\n    rows = wq.shape[0]\n    out = np.empty((h.shape[0], rows), dtype=np.float64)\n    for r0 in range(0, rows, rows_per_block):\n        w = dequant(")],
}

FUNCS = ("unpack", "fp16_values", "bf16_values", "dequant", "bf16_round", "logits_f64", "logits")


def _mutant(name):
    ns = {"np": np, "BLOCK": q4head.BLOCK, "topk_mapped": oracle.topk_mapped}
    for f in FUNCS:
        src = inspect.getsource(getattr(q4head, f))
        for old, new in MUTANTS[name]:
            src = src.replace(old, new)
        exec(compile(src, f"<mutant {name}: {f}>", "exec"), ns)
    return types.SimpleNamespace(**{f: ns[f] for f in FUNCS})


def test_every_substitution_applies():
    srcs = "".join(inspect.getsource(getattr(q4head, f)) for f in FUNCS)
    for name, subs in MUTANTS.items():
        for old, _ in subs:
            assert old in srcs, (name, old)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    m = _mutant(name)
    caught = []
    for pin in pins_q4.ALL_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_full_size_logits_spread():
    """The synthetic head at the page's size gives logits near N(0, 3^2) for
    N(0,1) hidden states (a check of the generator's scale range)."""
    import synth
    wq, sc = synth.q4_head(3, rows=4096)
    h = synth.hidden_states(4, 2)
    lg = q4head.logits_f64(h, wq, sc)
    assert 2.0 < lg.std() < 4.0
