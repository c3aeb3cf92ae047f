"""spec_round_noalloc: the round for callers that cannot let a library call
cudaMalloc (an engine that serves all device memory from its own pool, a
serving loop that cannot take cudaFree's device-wide synchronisation, a host
under a fixed memory budget).  Its scratch is a fixed device array inside
the library, shared by every call.

The test calls it through the C ABI twice in a row, on different inputs, and
checks each result bit for bit against spec_round (the allocating entry
point) and against the CPU oracle.  It lives in a file of its own that
pytest collects last, and it passes alone in a fresh process as well as
after the other tests.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g._load_build_module().build()
    import speculative_decoding_draft_column_gb300 as sd
    return sd


def _outputs(r, k):
    import torch
    cols, lanes, gamma = r.cols, r.lanes, r.gamma
    return (torch.full((cols, k), 0x1111, dtype=torch.int16, device="cuda"),
            torch.full((cols, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((lanes,), -7, dtype=torch.int32, device="cuda"),
            torch.full((lanes, gamma + 1), -7, dtype=torch.int32, device="cuda"))


def _call(sd, fn, r, k, x, t, d, outs):
    import torch
    sd.lib.spec_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    v, i, a, c = outs
    st = fn(x.data_ptr(), r.cols, r.V, k, v.data_ptr(), i.data_ptr(), t.data_ptr(), d.data_ptr(), r.lanes, r.gamma,
            a.data_ptr(), c.data_ptr())
    assert st == sd.SPEC_OK, sd.spec_last_error()
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("which", ["C2", "C1", "C5k64"])
def test_noalloc_matches_spec_round_twice_in_a_row(sd, which):
    if which == "C5k64":
        rounds = [synth.make_c5(seed=s, k=64, lanes=12, gamma=15, cols=90) for s in (41, 42)]
    else:
        rounds = [synth.CONFIGS[which](seed=s) for s in (31, 32)]
    for r in rounds:                       # two calls in a row, different inputs
        k = r.k
        x, t, d = gu.dev_u16(r.draft), gu.dev_u16(r.target), gu.dev_i32(r.drafts)
        want = _call(sd, sd.lib.spec_round, r, k, x, t, d, _outputs(r, k))
        got = _call(sd, sd.lib.spec_round_noalloc, r, k, x, t, d, _outputs(r, k))
        for g_, w_ in zip(got, want):
            assert np.array_equal(g_, w_)
        ov, oi = oracle.topk(r.draft, k)
        oa, oc = oracle.verify(r.target, r.drafts)
        assert np.array_equal(got[0].view(np.uint16), ov) and np.array_equal(got[1], oi)
        assert np.array_equal(got[2], oa) and np.array_equal(got[3], oc)
        assert got[2].tolist() == r.planted_accept.tolist()


def test_noalloc_rejects_sizes_beyond_its_limit(sd):
    P = 0x100000                             # never dereferenced: the size check fails first
    st = sd.lib.spec_round_noalloc(P, 8000, 1000, 8, P, P, P, P, 64, 7, P, P)
    assert st == sd.SPEC_ERR_ARG
    assert "8192" in sd.spec_last_error()
    st = sd.lib.spec_round_noalloc(P, 1, 1000, 8, P, P, P, P, 513, 1, P, P)
    assert st == sd.SPEC_ERR_ARG and "512" in sd.spec_last_error()
