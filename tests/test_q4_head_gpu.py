"""The Q4 shortlist head on the GPU against the oracle (oracle.q4head).

The logits: every one within the bound the arithmetic gives -- the kernel
sums each block of 64 products on the tensor cores in fp32, scales it and
adds it in fp32, then rounds once to bf16 -- of the exact value:

    |kernel - exact| <= 0.5 ulp_bf16(|exact| + E) + E,   E = 2^-16 * A,

A = sum_j |scale * (n_j - 8) * h_j|, the size of the terms any summation
order rounds (about 4x the worst case of 64 tensor-core additions and 80
fp32 FMAs at 2^-24 each).  Most logits equal the oracle's bf16 exactly.

The top-k: bit-exact, the pinned top-k oracle (shortlist ties by vocabulary
id) run on the kernel's own logits.  Needs a GPU.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from oracle import q4head
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g._load_build_module().build()
    oracle.load()
    import speculative_decoding_draft_column_gb300 as sd
    return sd


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def _device_head(sd, wq, sc):
    import torch
    rows, half = wq.shape
    d = 2 * half
    w = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(sc).view(np.int16)).cuda()
    wp = torch.empty_like(w)
    sp = torch.empty_like(s)
    sd.spec_shortlist_pack(w, s, rows, d, wp, sp)
    return wp, sp


def _check_logits(got_bits, hidden, wq, sc, what):
    x = q4head.logits_f64(hidden, wq, sc)
    a = q4head.abs_sum(hidden, wq, sc)
    k = q4head.bf16_values(got_bits)
    E = 2.0 ** -16 * a
    err = np.abs(k - x)
    bound = 0.5 * _ulp_bf16(np.abs(x) + E) + E
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} logits outside the bound; worst err/bound "
                           f"{float((err / bound).max()):.3f}")
    same = np.mean(got_bits == q4head.bf16_round(x))
    assert same > 0.99, f"{what}: only {same:.4f} of the logits equal the oracle's rounding"
    return float((err / bound).max())


@pytest.mark.parametrize("rows,d,cols", [(16, 64, 1), (64, 128, 3), (4096, 5120, 7), (2048, 5120, 17),
                                         (1024, 2048, 33)])
def test_logits_and_topk_small(sd, rows, d, cols):
    import torch
    wq, sc = synth.q4_head(21 + cols, rows=rows, d=d)
    h = synth.hidden_states(22 + cols, cols, d)
    wp, sp = _device_head(sd, wq, sc)
    hd = gu.dev_u16(h)
    lg = torch.full((cols, rows), 0x7F7F, dtype=torch.int16, device="cuda")
    k = min(8, rows)
    vals = torch.empty((cols, k), dtype=torch.int16, device="cuda")
    ids = torch.empty((cols, k), dtype=torch.int32, device="cuda")
    id_map = synth.shortlist_map(23, rows)
    sd.spec_shortlist_topk(hd, cols, d, wp, sp, rows, gu.dev_i32(id_map), k, lg, vals, ids)
    torch.cuda.synchronize()
    sd.spec_device_status()
    got = lg.cpu().numpy().view(np.uint16)
    _check_logits(got, h, wq, sc, f"rows={rows} d={d} cols={cols}")
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()),
                         oracle.topk_mapped(got, k, id_map), f"head top-k rows={rows} cols={cols}")


def test_logits_only_entry_matches(sd):
    import torch
    rows, d, cols = 512, 5120, 5
    wq, sc = synth.q4_head(31, rows=rows, d=d)
    h = synth.hidden_states(32, cols, d)
    wp, sp = _device_head(sd, wq, sc)
    lg = torch.empty((cols, rows), dtype=torch.int16, device="cuda")
    sd.spec_shortlist_logits(gu.dev_u16(h), cols, d, wp, sp, rows, lg)
    torch.cuda.synchronize()
    _check_logits(lg.cpu().numpy().view(np.uint16), h, wq, sc, "logits entry")


@pytest.mark.parametrize("cols", [7, 56])
def test_full_head(sd, cols):
    """The page's head: 131,072 rows of 5,120 weights (356.5 MB), k = 8, the
    drafter's 7 and 56 columns (one lane, eight lanes)."""
    import torch
    rows, d, k = synth.SHORTLIST, synth.HIDDEN, 8
    wq, sc = synth.q4_head(41)
    assert wq.nbytes + sc.nbytes == 356_515_840
    h = synth.hidden_states(42 + cols, cols, d)
    id_map = synth.shortlist_map(43)
    wp, sp = _device_head(sd, wq, sc)
    lg = torch.empty((cols, rows), dtype=torch.int16, device="cuda")
    vals = torch.empty((cols, k), dtype=torch.int16, device="cuda")
    ids = torch.empty((cols, k), dtype=torch.int32, device="cuda")
    sd.spec_shortlist_topk(gu.dev_u16(h), cols, d, wp, sp, rows, gu.dev_i32(id_map), k, lg, vals, ids)
    torch.cuda.synchronize()
    sd.spec_device_status()
    got = lg.cpu().numpy().view(np.uint16)
    pick = np.sort(synth.rng(44, cols).choice(cols, size=min(cols, 7), replace=False))
    _check_logits(got[pick], h[pick], wq, sc, f"full head cols={cols}")
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()),
                         oracle.topk_mapped(got, k, id_map), f"full head top-k cols={cols}")
