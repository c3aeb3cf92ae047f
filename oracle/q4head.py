"""CPU oracle of the Q4 shortlist head: logits of a 4-bit head, then the
mapped top-k ("A drafter inside the artifact", Ignis DFlash2 page, section
"How it works", second paragraph: an opt-in Q4 "shortlist" head over the
131,072 most frequent tokens, about 356 MB).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU legs are the only users.  The library never imports it.

The page gives the bit width, the row count and the size, not the layout.
The reading taken (the plainest one that gives the size):

* hidden width d (a multiple of 64; 5,120 gives the page's size);
* weights: uint8 [rows][d/2]; byte j of a row holds weight 2j in its low
  nibble and weight 2j+1 in its high nibble; a nibble n stands for n - 8;
* scales: fp16 bit patterns [rows][d/64]; scale b multiplies the block of
  weights 64b .. 64b+63 of its row;
* so 131,072 rows x (2,560 + 160) bytes = 356,515,840 bytes.

The logit of row i for a hidden state h (bf16, length d) is

    sum over blocks b of  scale[i][b] * sum over j in block b of (n_ij - 8) * h_j

computed here in float64 (every product is exact, and a sum of 5,120 such
terms keeps about 40 more bits than bf16 holds), then rounded once to bf16,
to nearest with ties to even, straight from the float64 value (no float32
step, so nothing is rounded twice).  The top-k of a column is then the
shortlist top-k: ties to the smaller vocabulary id id_map[i], output ids
are vocabulary ids (the pinned C oracle's topk_mapped).

No function here is unpinned: tests/pins_q4.py pins them by hand-worked
examples (tests/golden/q4head_examples.txt), closed forms (one-hot hidden
states pick one weight; constant weights sum h; zero scales give +0), and
the rounding cases that tell one rounding from another.
"""
from __future__ import annotations

import numpy as np

from . import topk_mapped

BLOCK = 64   # weights per scale


def unpack(wq: np.ndarray) -> np.ndarray:
    """Weights as integers n - 8, int8 [rows][2 * bytes per row]: element 2j
    from the low nibble of byte j, element 2j+1 from its high nibble."""
    b = np.ascontiguousarray(wq, dtype=np.uint8)
    rows, half = b.shape
    out = np.empty((rows, 2 * half), dtype=np.int8)
    out[:, 0::2] = (b & 0x0F).astype(np.int8) - 8
    out[:, 1::2] = (b >> 4).astype(np.int8) - 8
    return out


def fp16_values(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> float64 (exact)."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def dequant(wq: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The head as float64 [rows][d]: (n - 8) times its block's scale."""
    q = unpack(wq).astype(np.float64)
    rows, d = q.shape
    s = fp16_values(scales)
    assert s.shape == (rows, d // BLOCK), (s.shape, rows, d)
    return q * np.repeat(s, BLOCK, axis=1)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, to nearest, ties to even, in one step.
    A value v = m * 2^e (0.5 <= |m| < 1) keeps 8 significant bits: round
    m * 2^8 to an integer (numpy's rint rounds halves to even) and scale
    back; below the smallest normal the exponent stays at bf16's minimum
    (subnormals).  Overflow gives +-Inf."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)                      # bf16 normals have e >= -125 in frexp terms
    r = np.rint(np.ldexp(x, 8 - e))              # exact scaling by a power of two
    y = np.ldexp(r, e - 8)
    with np.errstate(over="ignore"):
        f = y.astype(np.float32)                 # exact: y has at most 8 significant bits
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    big = np.abs(y) >= 2.0 ** 128
    bits[big] = np.where(y[big] > 0, 0x7F80, 0xFF80).astype(np.uint16)
    return bits


def logits_f64(hidden: np.ndarray, wq: np.ndarray, scales: np.ndarray, rows_per_block: int = 2048) -> np.ndarray:
    """Exact-enough logits, float64 [cols][rows]; hidden: bf16 bits [cols][d]."""
    h = bf16_values(hidden)
    if h.ndim == 1:
        h = h[None, :]
    rows = wq.shape[0]
    out = np.empty((h.shape[0], rows), dtype=np.float64)
    for r0 in range(0, rows, rows_per_block):
        w = dequant(wq[r0:r0 + rows_per_block], scales[r0:r0 + rows_per_block])
        out[:, r0:r0 + rows_per_block] = h @ w.T
    return out


def logits(hidden: np.ndarray, wq: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The head's logits as bf16 bit patterns [cols][rows]."""
    return bf16_round(logits_f64(hidden, wq, scales))


def topk(hidden: np.ndarray, wq: np.ndarray, scales: np.ndarray, id_map: np.ndarray, k: int):
    """The head's logits, then the shortlist top-k of each column:
    (vals bf16 bits [cols][k], vocabulary ids [cols][k], logits bf16 bits)."""
    lg = logits(hidden, wq, scales)
    v, i = topk_mapped(lg, k, id_map)
    return v, i, lg


def abs_sum(hidden: np.ndarray, wq: np.ndarray, scales: np.ndarray, rows_per_block: int = 2048) -> np.ndarray:
    """sum over j of |scale * (n_ij - 8) * h_j| per (column, row): the scale of
    the rounding error any summation order can make (for tolerances)."""
    h = np.abs(bf16_values(hidden))
    if h.ndim == 1:
        h = h[None, :]
    rows = wq.shape[0]
    out = np.empty((h.shape[0], rows), dtype=np.float64)
    for r0 in range(0, rows, rows_per_block):
        w = np.abs(dequant(wq[r0:r0 + rows_per_block], scales[r0:r0 + rows_per_block]))
        out[:, r0:r0 + rows_per_block] = h @ w.T
    return out
