"""Sampled verify (speculative sampling with one-hot drafts, at T / top_p /
top_k as on the "A drafter inside the artifact" page, "The numbers"): the
oracle pinned by a hand-worked two-token column, its reduction to greedy
verify, softmax from a library routine, exact draw frequencies and
invariants."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.load()


def bf16(x: float) -> int:
    return int(synth.f32_to_bf16_bits(np.array([x], dtype=np.float32))[0])


def two_token_column(V: int = 16):
    """Token 3 has logit 2.0, token 9 has 1.0, every other token -30."""
    col = np.full(V, bf16(-30.0), dtype=np.uint16)
    col[3], col[9] = bf16(2.0), bf16(1.0)
    return col


def test_two_token_column_by_hand():
    col = two_token_column()
    vals, ids = oracle.topk(col[None, :], 2)
    kept, q = oracle.sampled_column(vals[0], ids[0], 1.0, 1.0)
    # softmax of (2, 1): e/(e+1) and 1/(e+1)
    assert kept == [3, 9]
    assert q[0] == pytest.approx(math.e / (math.e + 1), rel=1e-15)
    assert q[1] == pytest.approx(1 / (math.e + 1), rel=1e-15)
    # temperature 0.5 doubles the gap: e^2/(e^2+1)
    _, qh = oracle.sampled_column(vals[0], ids[0], 0.5, 1.0)
    assert qh[0] == pytest.approx(math.e ** 2 / (math.e ** 2 + 1), rel=1e-15)
    # draft = token 9 (q = 0.2689...): accepted below, rejected above; the
    # rejection draws from what is left, token 3
    assert oracle.sampled_decision(kept, q, 9, 0.25, 0.9)[:2] == (True, 9)
    assert oracle.sampled_decision(kept, q, 9, 0.30, 0.9)[:2] == (False, 3)
    # bonus position (no draft): running weight 0.731 then 1.0
    assert oracle.sampled_decision(kept, q, None, 0.0, 0.70)[:2] == (False, 3)
    assert oracle.sampled_decision(kept, q, None, 0.0, 0.80)[:2] == (False, 9)
    # top_p 0.7: the nucleus is token 3 alone (0.731 >= 0.7), so draft 9 is
    # never accepted and the draw is always token 3
    kept7, q7 = oracle.sampled_column(vals[0], ids[0], 1.0, 0.7)
    assert kept7 == [3] and q7 == [1.0]
    assert oracle.sampled_decision(kept7, q7, 9, 0.0, 0.99)[:2] == (False, 3)


def test_full_nucleus_is_softmax():
    """top_p = 1 and top_k = V: q is the softmax of logits / T (scipy)."""
    from scipy.special import softmax
    col = synth._draft_block(11, 1, 24, 2.0, quant=False)[0]
    vals, ids = oracle.topk(col[None, :], 24)
    for T in (0.5, 1.0, 1.7):
        kept, q = oracle.sampled_column(vals[0], ids[0], T, 1.0)
        logits = (col.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        want = softmax(logits / T)
        assert kept == list(ids[0])
        np.testing.assert_allclose(q, want[kept], rtol=1e-12)


def test_residual_draw_frequencies():
    """Over a fine grid of u2 the residual draw hits each kept token (draft
    removed) in proportion to its mass, to within one grid step."""
    col = synth._draft_block(12, 1, 64, 1.0, quant=False)[0]
    vals, ids = oracle.topk(col[None, :], 20)
    kept, q = oracle.sampled_column(vals[0], ids[0], 1.0, 0.95)
    draft = kept[1]
    N = 20000
    counts = {}
    for i in range(N):
        ok, tok, _ = oracle.sampled_decision(kept, q, draft, 1.0, (i + 0.5) / N)
        assert not ok and tok != draft and tok in kept
        counts[tok] = counts.get(tok, 0) + 1
    W = sum(qt for tok, qt in zip(kept, q) if tok != draft)
    for tok, qt in zip(kept, q):
        if tok == draft:
            continue
        assert abs(counts.get(tok, 0) / N - qt / W) <= 1.0 / N + 1e-12


def test_top_k_one_is_greedy_verify():
    """With top_k = 1 the target puts all mass on its argmax: every uniform
    gives the greedy result."""
    for seed, make in ((4, synth.make_c1), (5, synth.make_c3)):
        r = make(seed=seed, V=3000)
        u = synth.rng(40 + seed, 0).random((r.lanes, r.gamma + 1, 2))
        a, c, _ = oracle.sampled_verify(r.target, r.drafts, 1.0, 0.95, 1, u)
        ga, gc = oracle.verify(r.target, r.drafts)
        np.testing.assert_array_equal(a, ga)
        np.testing.assert_array_equal(c, gc)


def test_cold_temperature_is_greedy_verify():
    """T -> 0 concentrates the mass on the argmax (planted peaks 24 against
    noise below 19): greedy again."""
    r = synth.make_c2(seed=6, V=2000)
    u = synth.rng(46, 0).random((r.lanes, r.gamma + 1, 2))
    a, c, _ = oracle.sampled_verify(r.target, r.drafts, 1e-3, 0.95, 20, u)
    ga, gc = oracle.verify(r.target, r.drafts)
    np.testing.assert_array_equal(a, ga)
    np.testing.assert_array_equal(c, gc)


def test_invariants():
    r = synth.make_c2(seed=7, V=5000)
    u = synth.rng(47, 0).random((r.lanes, r.gamma + 1, 2))
    vals, ids = oracle.topk(r.target.reshape(r.lanes * (r.gamma + 1), -1), 20)
    a, c, m = oracle.sampled_verify(r.target, r.drafts, 1.0, 0.95, 20, u)
    assert m > 0
    for ln in range(r.lanes):
        assert 0 <= a[ln] <= r.gamma
        np.testing.assert_array_equal(c[ln, :a[ln]], r.drafts[ln, :a[ln]])        # accepted drafts
        assert c[ln, a[ln]] in ids[ln * (r.gamma + 1) + a[ln]]                      # a draw from the top-k
        if a[ln] < r.gamma:
            assert c[ln, a[ln]] != r.drafts[ln, a[ln]]                               # never the rejected draft
        assert (c[ln, a[ln] + 1:] == -1).all()
