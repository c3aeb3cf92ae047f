"""spec_round_host from several host threads at once: the call holds the
library until its stream has drained, and an area that a larger call
replaces stays allocated, so concurrent calls never copy into staging that
another thread has grown or freed.  Needs a GPU."""
from __future__ import annotations

import threading

import numpy as np
import pytest

import oracle
import synth

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


def _host_round(sd, r):
    vals = np.zeros((r.cols, r.k), dtype=np.uint16)
    ids = np.zeros((r.cols, r.k), dtype=np.int32)
    acc = np.zeros(r.lanes, dtype=np.int32)
    com = np.zeros((r.lanes, r.gamma + 1), dtype=np.int32)
    sd.spec_round_host(r.draft, r.cols, r.V, r.k, vals, ids, r.target, r.drafts, r.lanes, r.gamma, acc, com)
    return vals, ids, acc, com


def test_concurrent_host_rounds_while_staging_grows(sd):
    import torch
    sd.spec_release()                                   # start from no staging at all
    small = synth.make_c1(seed=61, V=20_000)
    growing = [synth.make_c2(seed=62 + i, V=30_000 * (i + 1)) for i in range(4)]
    want_small = (oracle.topk(small.draft, small.k), oracle.verify(small.target, small.drafts))
    want_grow = [(oracle.topk(r.draft, r.k), oracle.verify(r.target, r.drafts)) for r in growing]
    errors = []

    def worker(rounds, wants, reps):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            sd.spec_set_stream(s)
            for rep in range(reps):
                i = rep % len(rounds)
                v, d, a, c = _host_round(sd, rounds[i])
                (wv, wi), (wa, wc) = wants[i]
                if not (np.array_equal(v, wv) and np.array_equal(d, wi) and np.array_equal(a, wa)
                        and np.array_equal(c, wc)):
                    errors.append(f"round {i} repeat {rep} differs from the oracle")
        except Exception as e:                          # noqa: BLE001 - reported below
            errors.append(repr(e))

    ts = [threading.Thread(target=worker, args=([small], [want_small], 24)),
          threading.Thread(target=worker, args=(growing, want_grow, 8))]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in ts), "a host call did not return"
    assert not errors, errors
    sd.spec_device_status()
    sd.spec_release()
