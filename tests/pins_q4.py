"""Pins of the Q4 shortlist head oracle (``oracle.q4head``): things the
head's definition fixes without the oracle's own code.

* hand-worked examples (tests/golden/q4head_examples.txt), including the
  three rounding cases that tell one-step round-to-nearest-even from
  rounding through float32 or truncating;
* one-hot hidden states: the logit of row i is then one weight times its
  block's scale times the one value -- read straight from the packed bytes
  by index, with scales and values chosen so the product is exact in bf16;
* constant weights (+1 everywhere, unit scales): the logit is the plain sum
  of the hidden state;
* zero scales or a zero hidden state: every logit is +0;
* the size of the page's head: 131,072 rows of 5,120 weights occupy
  356,515,840 bytes in this layout (the page: "about 356 MB").

Each pin takes the module under test (the oracle, or a planted mutant of it).
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "q4head_examples.txt")


def _f16_bits(vals) -> np.ndarray:
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def _bf16_bits_exact(vals) -> np.ndarray:
    """bf16 bits of values that bf16 holds exactly (asserted)."""
    f = np.asarray(vals, dtype=np.float32)
    b = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    back = (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert np.array_equal(back, f), "value not exact in bf16"
    return b


def parse_golden():
    """[(d, h bits [d], [(bytes [d/2], scales fp16 bits, expect bits)])]"""
    out = []
    cur = None
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "example":
            d = int(tok[2].split("=")[1])
            cur = [d, None, []]
            out.append(cur)
        elif tok[0] == "h":
            d = cur[0]
            if tok[1] == "mod8":
                h = [(j % 8) + float(tok[2]) for j in range(d)]
            else:
                h = [0.0] * d
                for item in tok[1].split("=", 1)[1].split(","):
                    j, v = item.split(":")
                    h[int(j)] = float(v)
            cur[1] = _bf16_bits_exact(h)
        elif tok[0] == "row":
            d = cur[0]
            kv = dict(t.split("=", 1) for t in tok[1:])
            b = np.full(d // 2, int(kv["fill"], 16), dtype=np.uint8)
            for item in kv.get("set", "").split(",") if "set" in kv else []:
                j, v = item.split(":")
                b[int(j)] = int(v, 16)
            sc = _f16_bits([float(x) for x in kv["scales"].split(",")])
            cur[2].append((b, sc, int(kv["expect"], 16)))
    return out


def pin_golden(q4):
    ex = parse_golden()
    assert len(ex) == 4
    for d, h, rows in ex:
        wq = np.stack([r[0] for r in rows])
        sc = np.stack([r[1] for r in rows])
        got = q4.logits(h[None, :], wq, sc)[0]
        want = np.array([r[2] for r in rows], dtype=np.uint16)
        assert np.array_equal(got, want), (got, want)


def _simple_head(seed, rows, d):
    """Random nibbles; scales with at most 3 significant bits (so scale x
    weight x a power of two is exact in bf16)."""
    g = np.random.default_rng(seed)
    wq = g.integers(0, 256, size=(rows, d // 2), dtype=np.uint8)
    mant = g.choice([1.0, 1.25, 1.5, 1.75], size=(rows, d // 64))
    sc = _f16_bits(mant * np.exp2(g.integers(-6, 2, size=(rows, d // 64))))
    return wq, sc


def pin_one_hot(q4, rows=48, d=256):
    wq, sc = _simple_head(5, rows, d)
    s = np.asarray(sc, dtype=np.uint16).view(np.float16).astype(np.float64)
    for j in (0, 1, 63, 64, 65, 130, 255):
        for v in (1.0, -0.5, 4.0):
            h = np.zeros(d)
            h[j] = v
            got = q4.logits(_bf16_bits_exact(h)[None, :], wq, sc)[0]
            byte = wq[:, j // 2].astype(np.int64)
            n = (byte & 0xF) if j % 2 == 0 else (byte >> 4)
            want = _bf16_bits_exact(s[:, j // 64] * (n - 8) * v)
            # a product equal to zero is +0 in the sum of +0 terms, or -0; compare as numbers there
            zero = (n - 8) == 0
            assert np.array_equal(got[~zero], want[~zero]), (j, v)
            assert np.all((got[zero] & 0x7FFF) == 0), (j, v)


def pin_constant_weights(q4, d=320):
    wq = np.full((3, d // 2), 0x99, dtype=np.uint8)          # every weight +1
    sc = _f16_bits(np.ones((3, d // 64)))
    g = np.random.default_rng(9)
    h = g.integers(-4, 5, size=(2, d)).astype(np.float64)    # small integers: every sum exact
    got = q4.logits(_bf16_bits_exact(h), wq, sc)
    want = _bf16_bits_exact(np.repeat(h.sum(axis=1, keepdims=True), 3, axis=1))
    assert np.array_equal(got, want)


def pin_zeros(q4, d=192):
    g = np.random.default_rng(10)
    wq = g.integers(0, 256, size=(5, d // 2), dtype=np.uint8)
    h = _bf16_bits_exact(g.integers(-8, 9, size=(2, d)).astype(np.float64))
    got = q4.logits(h, wq, _f16_bits(np.zeros((5, d // 64))))
    assert np.all(got == 0), got
    got = q4.logits(np.zeros((1, d), dtype=np.uint16), wq, _f16_bits(np.ones((5, d // 64))))
    assert np.all(got == 0), got


def pin_page_size(q4):
    rows, d = 131_072, 5_120
    assert rows * (d // 2) + rows * (d // 64) * 2 == 356_515_840


ALL_PINS = [pin_golden, pin_one_hot, pin_constant_weights, pin_zeros, pin_page_size]
