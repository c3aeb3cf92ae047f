"""Pins for the oracle's sampled verify (speculative sampling with one-hot
drafts at T / top_p / top_k, as on the "A drafter inside the artifact" page,
"The numbers").

Each ``pin_*`` takes an implementation ``impl`` -- the ``oracle`` module, or
a namespace holding copies of its ``sampled_column``, ``sampled_decision``
and ``sampled_verify`` with one planted mistake -- and raises
``AssertionError`` on a mismatch.  ``test_sampled_oracle.py`` runs every pin
against the oracle; ``test_sampled_mutants.py`` requires that some pin fails
for every planted mistake.  Top-k lists and greedy verify come from the C
oracle, pinned on their own.

What pins what:

* a two-token column worked by hand (softmax of (2, 1), temperature, the
  nucleus cut, accept and residual draw);
* two tied tokens (q = 1/2 each), where the uniforms and top_p sit exactly
  on a decision boundary: accept only when u < q, draw the first token whose
  running weight exceeds u2 times the total, cut the nucleus at the first
  running sum that reaches top_p;
* two whole lanes worked by hand (each position's own uniforms, the
  rejection's draw, the bonus draw from the last column);
* scipy's softmax for the full nucleus (top_p = 1, top_k = V);
* residual-draw frequencies over a fine grid of u2 (draft removed);
* reductions to greedy verify: top_k = 1, and T -> 0 with planted peaks;
* invariants on a seeded round.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth


def bf16(x: float) -> int:
    return int(synth.f32_to_bf16_bits(np.array([x], dtype=np.float32))[0])


def _column(V: int, logits: dict) -> np.ndarray:
    """A column of V bf16 logits, -30 everywhere but at the given ids."""
    col = np.full(V, bf16(-30.0), dtype=np.uint16)
    for i, x in logits.items():
        col[i] = bf16(x)
    return col


def _approx(a: float, b: float, rel: float = 1e-15) -> bool:
    return abs(a - b) <= rel * max(abs(a), abs(b))


def pin_two_token_column_by_hand(impl):
    """Token 3 has logit 2.0, token 9 has 1.0."""
    col = _column(16, {3: 2.0, 9: 1.0})
    vals, ids = oracle.topk(col[None, :], 2)
    kept, q = impl.sampled_column(vals[0], ids[0], 1.0, 1.0)
    # softmax of (2, 1): e/(e+1) and 1/(e+1)
    assert kept == [3, 9]
    assert _approx(q[0], math.e / (math.e + 1)) and _approx(q[1], 1 / (math.e + 1))
    # temperature 0.5 doubles the gap: e^2/(e^2+1)
    _, qh = impl.sampled_column(vals[0], ids[0], 0.5, 1.0)
    assert _approx(qh[0], math.e ** 2 / (math.e ** 2 + 1))
    # draft = token 9 (q = 0.2689...): accepted below, rejected above; the
    # rejection draws from what is left, token 3
    assert impl.sampled_decision(kept, q, 9, 0.25, 0.9)[:2] == (True, 9)
    assert impl.sampled_decision(kept, q, 9, 0.30, 0.9)[:2] == (False, 3)
    # bonus position (no draft): running weight 0.731 then 1.0
    assert impl.sampled_decision(kept, q, None, 0.0, 0.70)[:2] == (False, 3)
    assert impl.sampled_decision(kept, q, None, 0.0, 0.80)[:2] == (False, 9)
    # top_p 0.7: the nucleus is token 3 alone (0.731 >= 0.7), so draft 9 is
    # never accepted and the draw is always token 3
    kept7, q7 = impl.sampled_column(vals[0], ids[0], 1.0, 0.7)
    assert kept7 == [3] and q7 == [1.0]
    assert impl.sampled_decision(kept7, q7, 9, 0.0, 0.99)[:2] == (False, 3)


def pin_tied_pair_on_the_boundaries(impl):
    """Tokens 3 and 9 tie at logit 1.0: p = (1/2, 1/2) exactly, token 3
    first (the smaller id)."""
    col = _column(16, {3: 1.0, 9: 1.0})
    vals, ids = oracle.topk(col[None, :], 2)
    kept, q = impl.sampled_column(vals[0], ids[0], 1.0, 1.0)
    assert kept == [3, 9] and q == [0.5, 0.5]
    # top_p = 1/2 is reached by the first token alone: the nucleus stops there
    kept_h, q_h = impl.sampled_column(vals[0], ids[0], 1.0, 0.5)
    assert kept_h == [3] and q_h == [1.0]
    # u = q(draft) exactly: not below it, so the draft is rejected
    assert impl.sampled_decision(kept, q, 9, 0.5, 0.0)[:2] == (False, 3)
    assert impl.sampled_decision(kept, q, 9, 0.5 - 2.0 ** -53, 0.0)[:2] == (True, 9)
    # bonus draw with u2 = 1/2: token 3's running weight 1/2 does not exceed
    # 1/2, token 9's (1) does
    assert impl.sampled_decision(kept, q, None, 0.0, 0.5)[:2] == (False, 9)
    assert impl.sampled_decision(kept, q, None, 0.0, 0.5 - 2.0 ** -53)[:2] == (False, 3)


def pin_hand_worked_lanes(impl):
    """Two lanes, gamma = 2, worked by hand.  Target columns 0 and 1 of each
    lane tie tokens 3 and 9 (q = 1/2 each), column 2 ties tokens 5 and 7;
    both lanes draft (3, 9); T = 1, top_p = 1, top_k = 2.
      lane 0: u = 0.25 < 1/2 accepts 3; u = 0.75 rejects 9, and the draw
              over what is left (token 3 alone, weight 1/2; u2 = 0.9 -> 0.45)
              is 3: accept 1, commit (3, 3, -1);
      lane 1: 0.25 accepts 3, 0.40 accepts 9, the bonus draw from column 2
              with u2 = 0.75 passes token 5 (running 1/2) and takes 7:
              accept 2, commit (3, 9, 7)."""
    V = 16
    tie39, tie57 = _column(V, {3: 1.0, 9: 1.0}), _column(V, {5: 1.0, 7: 1.0})
    target = np.stack([tie39, tie39, tie57, tie39, tie39, tie57])
    drafts = np.array([[3, 9], [3, 9]], dtype=np.int32)
    u = np.array([[[0.25, 0.9], [0.75, 0.9], [0.0, 0.0]],
                  [[0.25, 0.9], [0.40, 0.9], [0.0, 0.75]]])
    a, c, _ = impl.sampled_verify(target, drafts, 1.0, 1.0, 2, u)
    assert list(a) == [1, 2]
    assert c.tolist() == [[3, 3, -1], [3, 9, 7]]


def pin_full_nucleus_is_softmax(impl):
    """top_p = 1 and top_k = V: q is the softmax of logits / T (scipy)."""
    from scipy.special import softmax
    col = synth._draft_block(11, 1, 24, 2.0, quant=False)[0]
    vals, ids = oracle.topk(col[None, :], 24)
    for T in (0.5, 1.0, 1.7):
        kept, q = impl.sampled_column(vals[0], ids[0], T, 1.0)
        logits = (col.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        want = softmax(logits / T)
        assert kept == list(ids[0])
        np.testing.assert_allclose(q, want[kept], rtol=1e-12)


def pin_residual_draw_frequencies(impl):
    """Over a fine grid of u2 the residual draw hits each kept token (draft
    removed) in proportion to its mass, to within one grid step."""
    col = synth._draft_block(12, 1, 64, 1.0, quant=False)[0]
    vals, ids = oracle.topk(col[None, :], 20)
    kept, q = impl.sampled_column(vals[0], ids[0], 1.0, 0.95)
    draft = kept[1]
    N = 20000
    counts = {}
    for i in range(N):
        ok, tok, _ = impl.sampled_decision(kept, q, draft, 1.0, (i + 0.5) / N)
        assert not ok and tok != draft and tok in kept
        counts[tok] = counts.get(tok, 0) + 1
    W = sum(qt for tok, qt in zip(kept, q) if tok != draft)
    for tok, qt in zip(kept, q):
        if tok == draft:
            continue
        assert abs(counts.get(tok, 0) / N - qt / W) <= 1.0 / N + 1e-12


def pin_top_k_one_is_greedy_verify(impl):
    """With top_k = 1 the target puts all mass on its argmax: every uniform
    gives the greedy result (C3 lanes accept all 15 drafts, so the bonus
    column is covered too)."""
    for seed, make in ((4, synth.make_c1), (5, synth.make_c3)):
        r = make(seed=seed, V=3000)
        u = synth.rng(40 + seed, 0).random((r.lanes, r.gamma + 1, 2))
        a, c, _ = impl.sampled_verify(r.target, r.drafts, 1.0, 0.95, 1, u)
        ga, gc = oracle.verify(r.target, r.drafts)
        np.testing.assert_array_equal(a, ga)
        np.testing.assert_array_equal(c, gc)


def pin_cold_temperature_is_greedy_verify(impl):
    """T -> 0 concentrates the mass on the argmax (planted peaks 24 against
    noise below 19): greedy again."""
    r = synth.make_c2(seed=6, V=2000)
    u = synth.rng(46, 0).random((r.lanes, r.gamma + 1, 2))
    a, c, _ = impl.sampled_verify(r.target, r.drafts, 1e-3, 0.95, 20, u)
    ga, gc = oracle.verify(r.target, r.drafts)
    np.testing.assert_array_equal(a, ga)
    np.testing.assert_array_equal(c, gc)


def pin_invariants(impl):
    r = synth.make_c2(seed=7, V=5000)
    u = synth.rng(47, 0).random((r.lanes, r.gamma + 1, 2))
    vals, ids = oracle.topk(r.target.reshape(r.lanes * (r.gamma + 1), -1), 20)
    a, c, m = impl.sampled_verify(r.target, r.drafts, 1.0, 0.95, 20, u)
    assert m > 0
    for ln in range(r.lanes):
        assert 0 <= a[ln] <= r.gamma
        np.testing.assert_array_equal(c[ln, :a[ln]], r.drafts[ln, :a[ln]])        # accepted drafts
        assert c[ln, a[ln]] in ids[ln * (r.gamma + 1) + a[ln]]                      # a draw from the top-k
        if a[ln] < r.gamma:
            assert c[ln, a[ln]] != r.drafts[ln, a[ln]]                               # never the rejected draft
        assert (c[ln, a[ln] + 1:] == -1).all()


ALL_PINS = [
    pin_two_token_column_by_hand, pin_tied_pair_on_the_boundaries, pin_hand_worked_lanes, pin_full_nucleus_is_softmax,
    pin_residual_draw_frequencies, pin_top_k_one_is_greedy_verify, pin_cold_temperature_is_greedy_verify,
    pin_invariants,
]
