"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.load()`` or a
deliberately broken build of it) and raises ``AssertionError`` on a mismatch.
``test_oracle_pins.py`` runs every pin against the real oracle;
``test_oracle_mutants.py`` runs them against copies of the oracle with one
planted mistake each and requires that some pin fails for every mutant.

What pins what:

* an independent selector (k rounds of "scan for the largest value, first
  index wins, remove it"), written here in plain Python, on many tiny columns
  with few levels, and exhaustively for V <= 5 over 4 levels;
* closed forms: planted peaks, all-ties columns, the 64-level quantised
  columns by a scan over levels;
* library routines for the special cases: k = V is numpy's lexsort of
  (id, -value); k = 1 and the verify argmax are numpy's argmax (first max);
* hand-worked examples in ``tests/golden/``;
* invariants of a top-k and of a greedy verify on arbitrary bf16 patterns;
* acceptance lengths planted by the input generator.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# helpers (test side; no oracle code)
# ----------------------------------------------------------------------------

def val(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return synth.bf16_to_f32(bits).astype(np.float64)


def parse_value(tok: str) -> int:
    tok = tok.strip()
    if tok in ("inf", "+inf"):
        return 0x7F80
    if tok == "-inf":
        return 0xFF80
    if tok == "-0":
        return 0x8000
    return synth.bf16_bits(float(tok))


def select_by_extraction(col_bits: np.ndarray, k: int, tie_ids=None):
    """Independent selector: k times, take the largest remaining value; among
    equal values the smallest tie id; remove it."""
    vals = [float(v) for v in val(col_bits)]
    ties = list(range(len(vals))) if tie_ids is None else [int(t) for t in tie_ids]
    alive = [True] * len(vals)
    out_rows = []
    for _ in range(k):
        best = -1
        for i in range(len(vals)):
            if not alive[i]:
                continue
            if best < 0 or vals[i] > vals[best] or (vals[i] == vals[best] and ties[i] < ties[best]):
                best = i
        alive[best] = False
        out_rows.append(best)
    ids = [ties[r] for r in out_rows]
    return np.array([int(col_bits[r]) for r in out_rows], dtype=np.uint16), np.array(ids, dtype=np.int32)


def check_topk_invariants(x: np.ndarray, k: int, vals: np.ndarray, ids: np.ndarray, id_map=None):
    """Invariants every correct top-k output satisfies (brute-force checked)."""
    cols, V = x.shape
    tie = np.arange(V) if id_map is None else np.asarray(id_map, dtype=np.int64)
    inv = {int(t): i for i, t in enumerate(tie)}
    for c in range(cols):
        xv = val(x[c])
        rows = np.array([inv[int(i)] for i in ids[c]])
        assert len(set(ids[c].tolist())) == k, "ids not distinct"
        assert np.all(rows >= 0) and np.all(rows < V)
        assert np.array_equal(vals[c], x[c, rows]), "value is not the element's own bits"
        v = val(vals[c])
        assert np.all(v[:-1] >= v[1:]), "values not non-increasing"
        for r in range(k - 1):
            if v[r] == v[r + 1]:
                assert ids[c, r] < ids[c, r + 1], "ties not in ascending id order"
        last_v, last_id = v[-1], ids[c, -1]
        omitted = np.ones(V, dtype=bool)
        omitted[rows] = False
        assert not np.any(xv[omitted] > last_v), "an omitted element beats the last selected"
        eq = omitted & (xv == last_v)
        assert not np.any(tie[eq] < last_id), "an omitted tie has a smaller id"


# ----------------------------------------------------------------------------
# top-k pins
# ----------------------------------------------------------------------------

TINY_LEVELS = [float("-inf"), -1.5, -0.0, 0.0, 0.5, 2.0, float("inf")]


def pin_topk_bruteforce(lib, n_cols: int = 24000, seed: int = 11):
    g = synth.rng(seed, 1)
    for V in range(1, 13):
        levels = [TINY_LEVELS[i] for i in sorted(g.choice(len(TINY_LEVELS), size=4, replace=False))]
        x = synth.levels_block(seed * 100 + V, n_cols // 12, V, levels)
        for k in sorted({1, min(2, V), (V + 1) // 2, V}):
            vals, ids = oracle.topk(x, k, threads=2, lib=lib)
            for c in range(x.shape[0]):
                ev, ei = select_by_extraction(x[c], k)
                assert np.array_equal(vals[c], ev) and np.array_equal(ids[c], ei), (V, k, c, x[c])


def pin_topk_exhaustive(lib):
    levels = [0xFF80, 0x8000, 0x0000, synth.bf16_bits(3.0)]   # -inf, -0, +0, 3
    for V in range(1, 6):
        grid = np.array(np.meshgrid(*[np.arange(4)] * V, indexing="ij")).reshape(V, -1).T
        x = np.array(levels, dtype=np.uint16)[grid]
        for k in range(1, V + 1):
            vals, ids = oracle.topk(x, k, threads=2, lib=lib)
            for c in range(x.shape[0]):
                ev, ei = select_by_extraction(x[c], k)
                assert np.array_equal(vals[c], ev) and np.array_equal(ids[c], ei), (V, k, x[c])


def pin_topk_planted_peaks(lib, V: int = 4099, cols: int = 5):
    """Three peaks 24 > 22 > 20 above noise clipped at 19 are the top 3."""
    x = np.empty((cols, V), dtype=np.uint16)
    pos = []
    for c in range(cols):
        x[c] = synth.f32_to_bf16_bits(synth.noise_column(7, c, V, 3.0))
        p = synth.rng(7, 1000 + c).choice(V, size=3, replace=False)
        for h, q in zip((24.0, 22.0, 20.0), p):
            x[c, q] = synth.bf16_bits(h)
        pos.append(p)
    vals, ids = oracle.topk(x, 8, threads=2, lib=lib)
    for c in range(cols):
        assert ids[c, :3].tolist() == [int(q) for q in pos[c]]
        assert vals[c, :3].tolist() == [synth.bf16_bits(h) for h in (24.0, 22.0, 20.0)]


def pin_topk_all_ties(lib, V: int = 1000):
    g = synth.rng(8, 0)
    for trial in range(6):
        b = int(g.integers(0, 0x7F80))
        b |= int(g.integers(0, 2)) << 15
        x = np.full((1, V), b, dtype=np.uint16)
        for k in (1, 7, 64):
            vals, ids = oracle.topk(x, k, threads=1, lib=lib)
            assert ids[0].tolist() == list(range(k))
            assert np.all(vals[0] == b)
    # a column of zeros with random signs: all tie; values keep their own sign
    z = (synth.rng(8, 1).integers(0, 2, size=(1, V)) << 15).astype(np.uint16)
    vals, ids = oracle.topk(z, 20, threads=1, lib=lib)
    assert ids[0].tolist() == list(range(20))
    assert np.array_equal(vals[0], z[0, :20])


def pin_topk_level_scan(lib, V: int = 20011, cols: int = 4, k: int = 20):
    """64-level columns: scan levels from the top, ids ascending within a level."""
    x = synth._draft_block(3, cols, V, 3.0, quant=True)
    vals, ids = oracle.topk(x, k, threads=2, lib=lib)
    for c in range(cols):
        xv = val(x[c])
        exp = []
        for level in sorted(set(xv.tolist()), reverse=True):
            exp.extend(np.nonzero(xv == level)[0].tolist())
            if len(exp) >= k:
                break
        assert ids[c].tolist() == exp[:k]
        assert np.array_equal(vals[c], x[c, exp[:k]])


def pin_topk_full_sort_lexsort(lib):
    """k = V: the whole column ordered by (value desc, id asc) = numpy lexsort."""
    x = synth.random_bits_block(21, 40, 50)
    for V in (1, 2, 17, 50):
        xs = np.ascontiguousarray(x[:, :V])
        vals, ids = oracle.topk(xs, V, threads=2, lib=lib)
        for c in range(xs.shape[0]):
            order = np.lexsort((np.arange(V), -val(xs[c])))
            assert ids[c].tolist() == order.tolist()
            assert np.array_equal(vals[c], xs[c, order])


def pin_topk_k1_argmax(lib):
    """k = 1: numpy's argmax (returns the first maximum)."""
    x = np.concatenate([synth.random_bits_block(22, 50, 777),
                        synth.levels_block(23, 50, 777, [-1.0, 0.0, -0.0, 1.0])])
    vals, ids = oracle.topk(x, 1, threads=2, lib=lib)
    am = np.array([np.argmax(val(r)) for r in x])
    assert np.array_equal(ids[:, 0], am)
    assert np.array_equal(vals[:, 0], x[np.arange(x.shape[0]), am])


def pin_topk_invariants(lib):
    x = np.concatenate([synth.random_bits_block(24, 12, 3001),
                        synth.levels_block(25, 12, 3001, [-2.0, -0.0, 0.0, 1.0, 5.0])])
    for k in (1, 3, 20, 64):
        vals, ids = oracle.topk(x, k, threads=2, lib=lib)
        check_topk_invariants(x, k, vals, ids)


def _golden_topk():
    rows = []
    with open(os.path.join(GOLDEN, "topk_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, values, mp, ids, vals = [p.strip() for p in line.split("|")]
            rows.append((int(k), [parse_value(t) for t in values.split()],
                         None if mp == "-" else [int(t) for t in mp.split()],
                         [int(t) for t in ids.split()], [parse_value(t) for t in vals.split()]))
    return rows


def pin_topk_golden(lib):
    rows = _golden_topk()
    assert len(rows) >= 10
    for k, values, mp, eids, evals in rows:
        x = np.array([values], dtype=np.uint16)
        if mp is None:
            vals, ids = oracle.topk(x, k, threads=1, lib=lib)
        else:
            vals, ids = oracle.topk_mapped(x, k, np.array(mp, dtype=np.int32), threads=1, lib=lib)
        assert ids[0].tolist() == eids, (values, mp, ids[0], eids)
        assert vals[0].tolist() == evals, (values, mp, vals[0], evals)


def pin_mapped_identity(lib):
    x = synth.random_bits_block(26, 20, 300)
    for k in (1, 5, 64):
        a = oracle.topk(x, k, threads=2, lib=lib)
        b = oracle.topk_mapped(x, k, np.arange(300, dtype=np.int32), threads=2, lib=lib)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_mapped_bruteforce(lib, n_cols: int = 400):
    for V in (1, 3, 8, 12):
        x = synth.levels_block(27 + V, n_cols // 4, V, [-1.0, -0.0, 0.0, 2.0])
        m = synth.rng(28, V).permutation(1000)[:V].astype(np.int32)
        for k in sorted({1, (V + 1) // 2, V}):
            vals, ids = oracle.topk_mapped(x, k, m, threads=2, lib=lib)
            for c in range(x.shape[0]):
                ev, ei = select_by_extraction(x[c], k, tie_ids=m)
                assert np.array_equal(vals[c], ev) and np.array_equal(ids[c], ei), (V, k, x[c], m)


def pin_mapped_all_ties_reversed(lib, V: int = 500):
    x = np.full((2, V), synth.bf16_bits(1.25), dtype=np.uint16)
    m = np.arange(V - 1, -1, -1, dtype=np.int32) + 1000      # local i -> 1000 + V-1-i
    vals, ids = oracle.topk_mapped(x, 9, m, threads=1, lib=lib)
    assert ids[0].tolist() == [1000 + i for i in range(9)]


# ----------------------------------------------------------------------------
# verify pins
# ----------------------------------------------------------------------------

def _golden_verify():
    rows = []
    with open(os.path.join(GOLDEN, "verify_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            gamma, cols, drafts, acc, com = [p.strip() for p in line.split("|")]
            tc = [[parse_value(t) for t in c.split()] for c in cols.split(";")]
            rows.append((int(gamma), tc, [int(t) for t in drafts.split()], int(acc),
                         [int(t) for t in com.split()]))
    return rows


def pin_verify_golden(lib):
    rows = _golden_verify()
    assert len(rows) >= 8
    for gamma, tc, drafts, eacc, ecom in rows:
        assert len(tc) == gamma + 1
        t = np.array(tc, dtype=np.uint16)
        acc, com = oracle.verify(t, np.array([drafts], dtype=np.int32), threads=1, lib=lib)
        assert int(acc[0]) == eacc, (tc, drafts, acc, eacc)
        assert com[0].tolist() == ecom, (tc, drafts, com, ecom)


def pin_verify_planted(lib):
    for V, lanes, gamma in ((1, 4, 1), (5, 6, 3), (1000, 16, 7), (4097, 8, 15)):
        tgt, drafts, acc_p, t_arg = synth.planted_verify(31 + V, lanes, gamma, V)
        acc, com = oracle.verify(tgt, drafts, threads=2, lib=lib)
        assert np.array_equal(acc, acc_p)
        for l in range(lanes):
            a = int(acc_p[l])
            assert com[l, : a + 1].tolist() == t_arg[l, : a + 1].tolist()
            assert np.all(com[l, a + 1:] == -1)


def pin_verify_all_ties(lib, V: int = 300):
    for gamma in (1, 7, 15):
        lanes = 3
        t = np.full((lanes * (gamma + 1), V), synth.bf16_bits(-3.5), dtype=np.uint16)
        d = np.zeros((lanes, gamma), dtype=np.int32)
        d[1, 0] = 5                      # first draft wrong
        d[2, gamma - 1] = 1              # last draft wrong
        acc, com = oracle.verify(t, d, threads=1, lib=lib)
        assert acc.tolist() == [gamma, 0, gamma - 1]
        assert com[0].tolist() == [0] * (gamma + 1)
        assert com[1].tolist() == [0] + [-1] * gamma
        assert com[2].tolist() == [0] * gamma + [-1]


def pin_verify_invariants(lib):
    for V, lanes, gamma in ((7, 50, 3), (300, 20, 15), (64, 40, 1)):
        x = synth.levels_block(40 + V, lanes * (gamma + 1), V, [-1.0, 0.0, -0.0, 2.0])
        am = np.array([np.argmax(val(r)) for r in x]).reshape(lanes, gamma + 1)
        # drafts: copy the argmax with random breaks, so that many lengths occur
        g = synth.rng(41, V)
        d = am[:, :gamma].copy().astype(np.int32)
        brk = g.integers(0, gamma + 1, size=lanes)
        for l in range(lanes):
            if brk[l] < gamma:
                d[l, brk[l]] = (am[l, brk[l]] + 1 + g.integers(0, V - 1 if V > 1 else 1)) % max(V, 2)
        acc, com = oracle.verify(x, d, threads=2, lib=lib)
        for l in range(lanes):
            a = int(acc[l])
            assert 0 <= a <= gamma
            assert com[l, :a].tolist() == d[l, :a].tolist()
            assert com[l, a] == am[l, a]
            assert np.all(com[l, a + 1:] == -1)
            assert a == gamma or d[l, a] != am[l, a]
            assert a == min(int(brk[l]), gamma) or (V == 1)


def pin_argmax_numpy(lib):
    x = np.concatenate([synth.random_bits_block(50, 30, 999),
                        synth.levels_block(51, 30, 999, [0.0, -0.0, 1.0])])
    ids = oracle.argmax(x, threads=2, lib=lib)
    assert np.array_equal(ids, np.array([np.argmax(val(r)) for r in x]))


ALL_PINS = [
    pin_topk_golden, pin_topk_exhaustive, pin_topk_bruteforce, pin_topk_planted_peaks,
    pin_topk_all_ties, pin_topk_level_scan, pin_topk_full_sort_lexsort, pin_topk_k1_argmax,
    pin_topk_invariants, pin_mapped_identity, pin_mapped_bruteforce, pin_mapped_all_ties_reversed,
    pin_verify_golden, pin_verify_planted, pin_verify_all_ties, pin_verify_invariants,
    pin_argmax_numpy,
]
