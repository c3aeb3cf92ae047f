"""Seeded synthetic inputs for the draft-column selection step.

This module only *draws* inputs: bf16 logit matrices, draft token ids and
shortlist id maps, with the shapes and value distributions of the five
workloads below. It holds none of the selection arithmetic (no sorting, no
top-k, no argmax): where a workload needs a known answer (a target argmax to
plant an acceptance length, say) the answer is *planted* — a peak written at
a chosen position, far above the noise — and the planted position is
returned alongside the data.

Both the CPU oracle tests and the CUDA parity tests draw their inputs here;
neither side imports the other.

Recipe (one stream per column, so the bytes do not depend on chunking):

* random numbers come from numpy's counter-based Philox generator keyed by
  ``(seed, stream)``; every column (draft or target) and every planting
  decision has its own stream id;
* noise is ``sigma * N(0, 1)`` drawn in float32, clipped to ``±19`` (more than
  6 sigma for every workload here, so that the planted peaks 20 / 22 / 24
  are strict maxima by construction), then rounded to bf16 with
  round-to-nearest-even;
* bf16 values are carried as ``uint16`` bit patterns.

The workloads (sizes from the speculative-decoding pages: the vocabulary of
the drafter's output head is V = 248,046 tokens; a lane drafts 7 tokens, or
15 with a block size of 16; the opt-in shortlist head covers 131,072 tokens):

======  ==============================================================
``C1``  1 lane, 7 drafts: 7 draft columns, N(0,3) + 3 planted peaks
        (24, 22, 20) per column, k = 8; verify over 8 target columns with
        planted peaks; drafts match the target argmax for the first 4
        positions, so the accepted length is 4.
``C2``  8 lanes x 7 drafts = 56 draft columns N(0,3), k = 8; verify over
        8 lanes x 8 target columns (one planted peak of 24 each), accepted
        length per lane uniform in 0..7.
``C3``  1 lane, gamma 15: 15 draft columns N(0,3) quantised to 64 levels
        (heavy ties), k = 20; verify over 3 lanes x 16 target columns of the
        same quantisation whose top level (7.75) is planted as a tie group;
        lane 0 accepts all 15 drafts, lane 1 none, lane 2 a seeded number.
``C4``  64 lanes x 7 drafts = 448 draft columns: N(0,2), with 45 seeded
        columns given +12 on one seeded logit, k = 20; verify over 64 lanes
        x 8 target columns of the same mixture plus a planted peak of 24.
``C5``  256 lanes x 15 drafts = 3,840 draft columns N(0,3), k swept over
        {1, 8, 20, 64}; verify over 256 lanes x 16 target columns (planted
        peaks), accepted length uniform in 0..15.
``C5s`` shortlist: 3,840 x 131,072 columns N(0,3) whose local ids map to
        vocabulary ids through the first 131,072 entries of a seeded
        permutation of [0, 248,046).
======  ==============================================================
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

VOCAB = 248_046
SHORTLIST = 131_072
NOISE_CLIP = 19.0

# stream-id bases: one Philox stream per column / per planting decision
_S_DRAFT = 0
_S_TARGET = 1 << 24
_S_PLANT = 2 << 24
_S_MISC = 3 << 24


def rng(seed: int, stream: int) -> np.random.Generator:
    """Counter-based generator for one (seed, stream) pair."""
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, stream & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs here are finite (no NaN), so no NaN special case is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits(value: float) -> int:
    """bf16 bit pattern of a float that bf16 holds exactly (planting heights)."""
    b = int(f32_to_bf16_bits(np.array([value], dtype=np.float32))[0])
    back = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
    assert float(back) == float(value), f"{value} is not exact in bf16"
    return b


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for test-side checks)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def noise_column(seed: int, stream: int, n: int, sigma: float) -> np.ndarray:
    """sigma * N(0,1) in float32, clipped to +-NOISE_CLIP."""
    z = rng(seed, stream).standard_normal(n, dtype=np.float32)
    z *= np.float32(sigma)
    np.clip(z, -NOISE_CLIP, NOISE_CLIP, out=z)
    return z


def quantise_64(x: np.ndarray) -> np.ndarray:
    """clamp(round(4x), -32, 31) / 4: 64 levels {-8.00, -7.75, ..., 7.75}."""
    return (np.clip(np.rint(x * 4.0), -32, 31) / 4.0).astype(np.float32)


@dataclasses.dataclass
class Round:
    """One synthetic round: draft columns for top-k, target columns for verify."""

    name: str
    V: int
    k: int
    draft: np.ndarray                      # uint16 [cols, V] (bf16 bits)
    target: np.ndarray | None = None       # uint16 [lanes*(gamma+1), V_target]
    drafts: np.ndarray | None = None       # int32 [lanes, gamma]
    gamma: int = 0
    lanes: int = 0
    V_target: int = 0
    id_map: np.ndarray | None = None       # int32 [V] (shortlist variant)
    planted_accept: np.ndarray | None = None   # int32 [lanes]
    planted_argmax: np.ndarray | None = None   # int32 [lanes, gamma+1]
    planted_draft_top: np.ndarray | None = None  # int32 [cols, 3] (C1 peaks)

    @property
    def cols(self) -> int:
        return int(self.draft.shape[0])

    def logit_bytes(self) -> int:
        t = 0 if self.target is None else self.target.size * 2
        return self.draft.size * 2 + t


def content_hash(*arrays: np.ndarray) -> str:
    """sha256[:16] over the arrays' bytes (C order), hashed in place."""
    h = hashlib.sha256()
    for a in arrays:
        if a is None:
            continue
        h.update(memoryview(np.ascontiguousarray(a)).cast("B"))
    return h.hexdigest()[:16]


def _draft_block(seed, cols, V, sigma, stream0=_S_DRAFT, quant=False):
    out = np.empty((cols, V), dtype=np.uint16)
    for c in range(cols):
        z = noise_column(seed, stream0 + c, V, sigma)
        if quant:
            z = quantise_64(z)
        out[c] = f32_to_bf16_bits(z)
    return out


def _plant_drafts(seed, t_argmax, accept, V):
    """drafts[l][i] = t[l][i] for i < a, drafts[l][a] != t[l][a], rest random."""
    lanes, gp1 = t_argmax.shape
    gamma = gp1 - 1
    drafts = np.empty((lanes, gamma), dtype=np.int32)
    for l in range(lanes):
        g = rng(seed, _S_MISC + 1000 + l)
        row = g.integers(0, V, size=gamma, dtype=np.int64)
        a = int(accept[l])
        row[:a] = t_argmax[l, :a]
        if a < gamma:
            # any id but the target's; with V == 1 an out-of-range id (never matches)
            row[a] = (t_argmax[l, a] + 1 + g.integers(0, V - 1)) % V if V > 1 else V
        drafts[l] = row.astype(np.int32)
    return drafts


def _target_with_peaks(seed, n_cols, V, sigma, height=24.0, quant=False):
    """Target columns: noise plus one planted strict maximum per column."""
    tgt = np.empty((n_cols, V), dtype=np.uint16)
    pos = np.empty(n_cols, dtype=np.int64)
    hb = bf16_bits(height)
    for t in range(n_cols):
        z = noise_column(seed, _S_TARGET + t, V, sigma)
        if quant:
            z = quantise_64(z)
        tgt[t] = f32_to_bf16_bits(z)
        p = int(rng(seed, _S_PLANT + t).integers(0, V))
        tgt[t, p] = hb
        pos[t] = p
    return tgt, pos


def make_c1(seed: int = 1, V: int = VOCAB) -> Round:
    cols, k, lanes, gamma = 7, 8, 1, 7
    draft = _draft_block(seed, cols, V, 3.0)
    heights = [bf16_bits(24.0), bf16_bits(22.0), bf16_bits(20.0)]
    top = np.empty((cols, 3), dtype=np.int32)
    for c in range(cols):
        p = rng(seed, _S_PLANT + 500_000 + c).choice(V, size=3, replace=False)
        for j in range(3):
            draft[c, p[j]] = heights[j]
        top[c] = p
    # target: same distribution with the same three planted heights
    tgt = _draft_block(seed, lanes * (gamma + 1), V, 3.0, stream0=_S_TARGET)
    t_arg = np.empty((lanes, gamma + 1), dtype=np.int32)
    for t in range(lanes * (gamma + 1)):
        p = rng(seed, _S_PLANT + t).choice(V, size=3, replace=False)
        for j in range(3):
            tgt[t, p[j]] = heights[j]
        t_arg.flat[t] = p[0]
    accept = np.array([4], dtype=np.int32)
    drafts = _plant_drafts(seed, t_arg, accept, V)
    return Round("C1", V, k, draft, tgt, drafts, gamma, lanes, V, None, accept, t_arg, top)


def make_c2(seed: int = 2, V: int = VOCAB, lanes: int = 8, gamma: int = 7) -> Round:
    cols, k = lanes * gamma, 8
    draft = _draft_block(seed, cols, V, 3.0)
    tgt, pos = _target_with_peaks(seed, lanes * (gamma + 1), V, 3.0)
    t_arg = pos.reshape(lanes, gamma + 1).astype(np.int32)
    accept = rng(seed, _S_MISC).integers(0, gamma + 1, size=lanes).astype(np.int32)
    drafts = _plant_drafts(seed, t_arg, accept, V)
    return Round("C2", V, k, draft, tgt, drafts, gamma, lanes, V, None, accept, t_arg)


def make_c3(seed: int = 3, V: int = VOCAB, ties: int = 4) -> Round:
    cols, k, lanes, gamma = 15, 20, 3, 15
    draft = _draft_block(seed, cols, V, 3.0, quant=True)
    n_t = lanes * (gamma + 1)
    top_bits = bf16_bits(7.75)
    below = bf16_bits(7.5)
    tgt = np.empty((n_t, V), dtype=np.uint16)
    t_arg = np.empty((lanes, gamma + 1), dtype=np.int32)
    for t in range(n_t):
        z = quantise_64(noise_column(seed, _S_TARGET + t, V, 3.0))
        col = f32_to_bf16_bits(z)
        col[col == top_bits] = below          # top level emptied ...
        p = np.sort(rng(seed, _S_PLANT + t).choice(V, size=ties, replace=False))
        col[p] = top_bits                     # ... then planted as a tie group
        tgt[t] = col
        t_arg.flat[t] = p[0]                  # ties go to the smallest id
    a2 = int(rng(seed, _S_MISC).integers(1, gamma))
    accept = np.array([gamma, 0, a2], dtype=np.int32)
    drafts = _plant_drafts(seed, t_arg, accept, V)
    return Round("C3", V, k, draft, tgt, drafts, gamma, lanes, V, None, accept, t_arg)


def _mixture_block(seed, cols, V, stream0, frac=0.10):
    out = np.empty((cols, V), dtype=np.uint16)
    n_peaked = int(round(frac * cols))
    peaked = set(rng(seed, stream0 + (1 << 22)).choice(cols, size=n_peaked, replace=False).tolist())
    for c in range(cols):
        z = noise_column(seed, stream0 + c, V, 2.0)
        if c in peaked:
            p = int(rng(seed, stream0 + (1 << 23) + c).integers(0, V))
            z[p] += np.float32(12.0)
        out[c] = f32_to_bf16_bits(z)
    return out


def make_c4(seed: int = 4, V: int = VOCAB, lanes: int = 64, gamma: int = 7) -> Round:
    cols, k = lanes * gamma, 20
    draft = _mixture_block(seed, cols, V, _S_DRAFT)
    n_t = lanes * (gamma + 1)
    tgt = _mixture_block(seed, n_t, V, _S_TARGET)
    hb = bf16_bits(24.0)
    t_arg = np.empty((lanes, gamma + 1), dtype=np.int32)
    for t in range(n_t):
        p = int(rng(seed, _S_PLANT + t).integers(0, V))
        tgt[t, p] = hb
        t_arg.flat[t] = p
    accept = rng(seed, _S_MISC).integers(0, gamma + 1, size=lanes).astype(np.int32)
    drafts = _plant_drafts(seed, t_arg, accept, V)
    return Round("C4", V, k, draft, tgt, drafts, gamma, lanes, V, None, accept, t_arg)


def make_c5(seed: int = 5, V: int = VOCAB, k: int = 8, lanes: int = 256, gamma: int = 15,
            cols: int | None = None, verify: bool = True) -> Round:
    cols = lanes * gamma if cols is None else cols
    draft = _draft_block(seed, cols, V, 3.0)
    r = Round("C5", V, k, draft)
    if verify:
        tgt, pos = _target_with_peaks(seed, lanes * (gamma + 1), V, 3.0)
        t_arg = pos.reshape(lanes, gamma + 1).astype(np.int32)
        accept = rng(seed, _S_MISC).integers(0, gamma + 1, size=lanes).astype(np.int32)
        r.target, r.gamma, r.lanes, r.V_target = tgt, gamma, lanes, V
        r.drafts = _plant_drafts(seed, t_arg, accept, V)
        r.planted_accept, r.planted_argmax = accept, t_arg
    return r


def shortlist_map(seed: int, V_local: int = SHORTLIST, vocab: int = VOCAB) -> np.ndarray:
    """First V_local entries of a seeded permutation of [0, vocab)."""
    perm = rng(seed, _S_MISC + 7).permutation(vocab)
    return perm[:V_local].astype(np.int32)


def make_c5s(seed: int = 6, k: int = 8, cols: int = 3840, V_local: int = SHORTLIST) -> Round:
    draft = _draft_block(seed, cols, V_local, 3.0)
    r = Round("C5s", V_local, k, draft)
    r.id_map = shortlist_map(seed, V_local)
    return r


CONFIGS = {"C1": make_c1, "C2": make_c2, "C3": make_c3, "C4": make_c4, "C5": make_c5, "C5s": make_c5s}


# ----------------------------------------------------------------------------
# small / edge-case generators (parity sweeps)
# ----------------------------------------------------------------------------

def levels_block(seed: int, cols: int, V: int, levels: list[float], stream0: int = _S_MISC + 50_000) -> np.ndarray:
    """Columns whose values are drawn uniformly from a few bf16 levels (ties)."""
    lv = np.array([bf16_bits(x) if np.isfinite(x) else (0x7F80 if x > 0 else 0xFF80) for x in levels],
                  dtype=np.uint16)
    out = np.empty((cols, V), dtype=np.uint16)
    for c in range(cols):
        out[c] = lv[rng(seed, stream0 + c).integers(0, len(lv), size=V)]
    return out


def signed_zero_bits() -> tuple[int, int]:
    return 0x0000, 0x8000


def random_bits_block(seed: int, cols: int, V: int, stream0: int = _S_MISC + 90_000) -> np.ndarray:
    """Arbitrary non-NaN bf16 bit patterns (every finite value, ±0, ±Inf)."""
    out = np.empty((cols, V), dtype=np.uint16)
    for c in range(cols):
        b = rng(seed, stream0 + c).integers(0, 1 << 16, size=V, dtype=np.uint32).astype(np.uint16)
        nan = (b & 0x7FFF) > 0x7F80
        b[nan] = b[nan] & 0x807F          # fold NaN patterns onto finite ones
        out[c] = b
    return out


def random_drafts(seed: int, lanes: int, gamma: int, V: int) -> np.ndarray:
    return rng(seed, _S_MISC + 70_000).integers(0, V, size=(lanes, gamma)).astype(np.int32)


def planted_verify(seed: int, lanes: int, gamma: int, V: int, sigma: float = 3.0,
                   accept: np.ndarray | None = None):
    """Target columns with planted argmax and drafts planted to a known length."""
    tgt, pos = _target_with_peaks(seed, lanes * (gamma + 1), V, sigma)
    t_arg = pos.reshape(lanes, gamma + 1).astype(np.int32)
    if accept is None:
        accept = rng(seed, _S_MISC).integers(0, gamma + 1, size=lanes).astype(np.int32)
    drafts = _plant_drafts(seed, t_arg, accept, V)
    return tgt, drafts, np.asarray(accept, dtype=np.int32), t_arg


# ----------------------------------------------------------------------------
# Q4 shortlist head (weights, scales, hidden states)
# ----------------------------------------------------------------------------

HIDDEN = 5120           # hidden width that gives the head's size: 131,072 x (2,560 + 160) B = 356.5 MB
_S_HEAD = 4 << 24


def q4_head(seed: int, rows: int = SHORTLIST, d: int = HIDDEN, scale_lo: float = 0.006,
            scale_hi: float = 0.012, rows_per_stream: int = 4096):
    """A synthetic Q4 head: packed nibbles uint8 [rows][d/2] (uniform bytes:
    every nibble 0..15, i.e. weights -8..7) and fp16 scale bit patterns
    [rows][d/64] uniform in [scale_lo, scale_hi] (rounded to fp16).  With
    N(0,1) hidden states the logits come out near N(0, 3^2).  One Philox
    stream per block of rows."""
    assert d % 64 == 0
    wq = np.empty((rows, d // 2), dtype=np.uint8)
    sc = np.empty((rows, d // 64), dtype=np.uint16)
    for r0 in range(0, rows, rows_per_stream):
        r1 = min(rows, r0 + rows_per_stream)
        g = rng(seed, _S_HEAD + r0 // rows_per_stream)
        wq[r0:r1] = g.integers(0, 256, size=(r1 - r0, d // 2), dtype=np.uint8)
        s = g.uniform(scale_lo, scale_hi, size=(r1 - r0, d // 64)).astype(np.float16)
        sc[r0:r1] = s.view(np.uint16)
    return wq, sc


def hidden_states(seed: int, cols: int, d: int = HIDDEN) -> np.ndarray:
    """bf16 bit patterns [cols][d], N(0,1) rounded to bf16 (RNE)."""
    out = np.empty((cols, d), dtype=np.uint16)
    for c in range(cols):
        out[c] = f32_to_bf16_bits(rng(seed, _S_HEAD + (1 << 20) + c).standard_normal(d, dtype=np.float32))
    return out
