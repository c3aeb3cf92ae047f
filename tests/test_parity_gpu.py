"""CUDA path vs the CPU oracle, element by element and bit-exact: top-k ids and
bf16 bits, accept lengths and committed ids.  Every call goes through the C
ABI (via the thin binding), once on each streaming kernel.  Needs a GPU."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g
    g._load_build_module().build()
    oracle.load()
    import speculative_decoding_draft_column_gb300 as sd
    return sd


@pytest.fixture(autouse=True, params=[1, 2, 3], ids=["warp", "cta", "gm"])
def kernel(request, _lib):
    """Every parity case runs on each streaming kernel (forced), whatever the
    automatic choice would be for its size (the group-maxima kernel hands
    columns shorter than 4096 to the CTA kernel)."""
    _lib.spec_set_kernel(request.param)
    yield request.param
    _lib.spec_set_kernel(_lib.SPEC_KERNEL_AUTO)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
def test_workload_full_size(name):
    r = synth.CONFIGS[name]()
    want_t = oracle.topk(r.draft, r.k)
    want_v = oracle.verify(r.target, r.drafts)
    gu.assert_topk_equal(gu.run_topk(r.draft, r.k), want_t, f"{name} spec_topk")
    gu.assert_verify_equal(gu.run_verify(r.target, r.drafts), want_v, f"{name} spec_verify")
    v, i, a, c = gu.run_round(r.draft, r.k, r.target, r.drafts)
    gu.assert_topk_equal((v, i), want_t, f"{name} spec_round top-k")
    gu.assert_verify_equal((a, c), want_v, f"{name} spec_round verify")
    assert want_v[0].tolist() == r.planted_accept.tolist()
    if r.planted_draft_top is not None:
        assert np.array_equal(i[:, :3], r.planted_draft_top)


@pytest.mark.parametrize("k", [1, 8, 20, 64])
def test_c5_k_sweep_reduced(k):
    r = synth.make_c5(k=k, lanes=24, gamma=15, cols=480)
    gu.assert_topk_equal(gu.run_topk(r.draft, k), oracle.topk(r.draft, k), f"C5 k={k}")
    v, i, a, c = gu.run_round(r.draft, k, r.target, r.drafts)
    gu.assert_topk_equal((v, i), oracle.topk(r.draft, k), f"C5 round k={k}")
    gu.assert_verify_equal((a, c), oracle.verify(r.target, r.drafts), f"C5 round verify k={k}")
    assert a.tolist() == r.planted_accept.tolist()


def _torch_topk_properties(x_dev, V, k, vals, ids):
    """Properties that hold at any size, checked on the device for every
    column: ids distinct and in range, values are the elements' own bits,
    non-increasing, ties ascending, and nothing omitted beats the last one."""
    import torch
    cols = x_dev.shape[0]
    idl = ids.long()
    assert int(idl.min()) >= 0 and int(idl.max()) < V
    srt = torch.sort(idl, dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all()), "duplicate ids"
    got_bits = torch.gather(x_dev, 1, idl)
    assert torch.equal(got_bits, vals), "values are not the selected elements' bits"
    xf = (x_dev.to(torch.int32) & 0xFFFF).bitwise_left_shift(16).view(torch.float32)
    vf = (vals.to(torch.int32) & 0xFFFF).bitwise_left_shift(16).view(torch.float32)
    assert bool((vf[:, 1:] <= vf[:, :-1]).all()), "values not non-increasing"
    tie = vf[:, 1:] == vf[:, :-1]
    assert bool(((idl[:, 1:] > idl[:, :-1]) | ~tie).all()), "ties not in ascending id order"
    last = vf[:, -1:]
    gt = (xf > last).sum(dim=1)
    assert bool((gt <= k - 1).all()), "an element above the last selected value was omitted"
    eq_before = ((xf == last) & (torch.arange(V, device=x_dev.device)[None, :] < idl[:, -1:])).sum(dim=1)
    sel_eq_before = ((vf == last) & (idl < idl[:, -1:])).sum(dim=1)
    assert torch.equal(eq_before, sel_eq_before), "an omitted tie has a smaller id"
    del cols


@pytest.fixture(scope="module")
def c5_inputs():
    """The full C5 round (3,840 draft columns, 256 lanes x 16 target columns,
    V = 248,046), drawn once and kept on the device for every k and kernel."""
    r = synth.make_c5(k=8)
    x, t = gu.dev_u16(r.draft), gu.dev_u16(r.target)
    want_v = oracle.verify(r.target, r.drafts)
    assert want_v[0].tolist() == r.planted_accept.tolist()
    return r, x, t, gu.dev_i32(r.drafts), want_v


@pytest.mark.parametrize("k", [1, 8, 20, 64])
def test_c5_full_size_sampled(c5_inputs, k):
    """The whole C5 round in one launch at every k of the sweep: every column
    checked by properties on the device, 64 seeded columns and every verify
    lane against the oracle."""
    import torch
    sd = gu.sd_module()
    r, x, t, d, (wa, wc) = c5_inputs
    cols, V = r.cols, r.V
    vals = torch.full((cols, k), 0x5A5A, dtype=torch.int16, device="cuda")
    ids = torch.full((cols, k), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((r.lanes,), -7, dtype=torch.int32, device="cuda")
    com = torch.full((r.lanes, r.gamma + 1), -7, dtype=torch.int32, device="cuda")
    sd.spec_round(x, cols, V, k, vals, ids, t, d, r.lanes, r.gamma, acc, com)
    torch.cuda.synchronize()
    sd.spec_device_status()
    for c0 in range(0, cols, 256):
        _torch_topk_properties(x[c0:c0 + 256], V, k, vals[c0:c0 + 256], ids[c0:c0 + 256])
    pick = np.sort(synth.rng(99, k).choice(cols, size=64, replace=False))
    wv, wi = oracle.topk(r.draft[pick], k)
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16)[pick], ids.cpu().numpy()[pick]), (wv, wi),
                         f"C5 k={k} sampled columns")
    gu.assert_verify_equal((acc.cpu().numpy(), com.cpu().numpy()), (wa, wc), f"C5 k={k} verify")


@pytest.mark.parametrize("k", [1, 8, 20, 64])
def test_c5_shortlist_reduced(k):
    r = synth.make_c5s(k=k, cols=384)
    got = gu.run_topk(r.draft, k, id_map=r.id_map)
    gu.assert_topk_equal(got, oracle.topk_mapped(r.draft, k, r.id_map), f"C5s k={k}")


@pytest.fixture(scope="module")
def c5s_inputs():
    """The full shortlist round (3,840 x 131,072 columns and the id map),
    drawn once and kept on the device."""
    r = synth.make_c5s(k=8)
    return r, gu.dev_u16(r.draft), gu.dev_i32(r.id_map)


@pytest.mark.parametrize("k", [1, 8, 20, 64])
def test_c5_shortlist_full_size_sampled(c5s_inputs, k):
    """spec_topk_mapped on the full shortlist round at every k: 96 seeded
    columns against the oracle, and every column: ids in the map's image,
    values the mapped elements' own bits, non-increasing."""
    import torch
    sd = gu.sd_module()
    r, x, m = c5s_inputs
    cols, V = r.cols, r.V
    vals = torch.full((cols, k), 0x5A5A, dtype=torch.int16, device="cuda")
    ids = torch.full((cols, k), -7, dtype=torch.int32, device="cuda")
    sd.spec_topk_mapped(x, cols, V, k, m, vals, ids)
    torch.cuda.synchronize()
    sd.spec_device_status()
    pick = np.sort(synth.rng(98, k).choice(cols, size=96, replace=False))
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16)[pick], ids.cpu().numpy()[pick]),
                         oracle.topk_mapped(r.draft[pick], k, r.id_map), f"C5s k={k} sampled columns")
    inv = torch.full((synth.VOCAB,), -1, dtype=torch.int64, device="cuda")
    inv[m.long()] = torch.arange(V, device="cuda")
    loc = inv[ids.long()]
    assert int(loc.min()) >= 0
    assert torch.equal(torch.gather(x, 1, loc), vals)
    vf = (vals.to(torch.int32) & 0xFFFF).bitwise_left_shift(16).view(torch.float32)
    assert bool((vf[:, 1:] <= vf[:, :-1]).all())


@pytest.mark.parametrize("name", ["C1", "C2"])
def test_spec_verify_fixed_vocabulary(name):
    """spec_verify, the call with no V argument (it runs over the pages'
    248,046-token vocabulary), on the C1 and C2 target columns."""
    import torch
    sd = gu.sd_module()
    r = synth.CONFIGS[name]()
    assert r.V == sd.SPEC_VOCAB
    t = gu.dev_u16(r.target, 3)
    acc = gu.Guarded(r.lanes, torch.int32)
    com = gu.Guarded(r.lanes * (r.gamma + 1), torch.int32)
    sd.spec_verify(t, gu.dev_i32(r.drafts), r.lanes, r.gamma, acc.view, com.view)
    torch.cuda.synchronize()
    sd.spec_device_status()
    acc.check_guards()
    com.check_guards()
    got = (acc.host(), com.host().reshape(r.lanes, r.gamma + 1))
    gu.assert_verify_equal(got, oracle.verify(r.target, r.drafts), f"{name} spec_verify")
    assert got[0].tolist() == r.planted_accept.tolist()


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

EDGE_V = [1, 2, 7, 8, 9, 15, 16, 17, 255, 256, 257, 2047, 2048, 2049, 65535, 65536, 65537, 131072, 248046]
EDGE_K = [1, 2, 7, 8, 20, 32, 33, 64]


def _edge_block(kind: int, seed: int, cols: int, V: int) -> np.ndarray:
    if kind == 0:
        return synth.random_bits_block(seed, cols, V)
    if kind == 1:
        return synth.levels_block(seed, cols, V, [-1.0, -0.0, 0.0, 3.0, float("inf")])
    if kind == 2:
        return np.full((cols, V), synth.bf16_bits(-2.25), dtype=np.uint16)
    return synth._draft_block(seed, cols, V, 3.0, quant=True)


@pytest.mark.parametrize("V", EDGE_V)
def test_topk_edge_sweep(V):
    n = 0
    for k in EDGE_K + [V]:
        if k > V or k > 64:
            continue
        for cols in (1, 7):
            kind = (n + V) % 4
            off = (n * 3 + V) % 8
            x = _edge_block(kind, 1000 + n + V, cols, V)
            gu.assert_topk_equal(gu.run_topk(x, k, offset=off), oracle.topk(x, k),
                                 f"V={V} k={k} cols={cols} kind={kind} offset={off}")
            n += 1


@pytest.mark.parametrize("offset", range(8))
def test_every_16_byte_phase(offset):
    x = synth.random_bits_block(77 + offset, 9, 20_011)
    gu.assert_topk_equal(gu.run_topk(x, 20, offset=offset), oracle.topk(x, 20), f"offset {offset}")


def test_many_columns_tiny_v():
    x = synth.levels_block(5, 3000, 5, [0.0, 1.0, -0.0])
    gu.assert_topk_equal(gu.run_topk(x, 3), oracle.topk(x, 3), "3000 x 5")


def test_ties_everywhere_large():
    x = np.full((56, 248_046), synth.bf16_bits(1.5), dtype=np.uint16)
    for k in (1, 8, 64):
        v, i = gu.run_topk(x, k)
        assert np.all(i == np.arange(k)[None, :]) and np.all(v == synth.bf16_bits(1.5))


def test_argmax_ties_column_mode():
    """128 columns of 65,536 logits from three levels, the maximum repeated in
    nearly every group of 64: enough columns for the group-maxima kernel's
    column mode, whose k = 1 finish must return the first position at the
    maximum (top-1, and greedy verify of 16 lanes)."""
    V = 65_536
    x = synth.levels_block(31, 128, V, [0.0, 1.0, -0.0])
    gu.assert_topk_equal(gu.run_topk(x, 1), oracle.topk(x, 1), "top-1 ties, 128 columns")
    lanes, gamma = 16, 7
    t = synth.levels_block(32, lanes * (gamma + 1), V, [0.0, 2.0, 1.0])
    d = synth.random_drafts(33, lanes, gamma, V)
    am = oracle.argmax(t).reshape(lanes, gamma + 1)
    d[: lanes // 2] = am[: lanes // 2, :gamma]   # half the lanes accept every draft
    gu.assert_verify_equal(gu.run_verify(t, d), oracle.verify(t, d), "verify ties, 128 columns")


def test_signed_zero_and_inf():
    V = 70_001
    x = np.full((4, V), 0xFF80, dtype=np.uint16)                  # all -inf
    g = synth.rng(3, 3)
    for c in range(4):
        p = g.choice(V, size=40, replace=False)
        x[c, p[:20]] = 0x8000                                     # -0
        x[c, p[20:]] = 0x0000                                     # +0
    x[3, 12345] = 0x7F80                                          # one +inf
    for k in (1, 20, 41, 64):
        gu.assert_topk_equal(gu.run_topk(x, k), oracle.topk(x, k), f"zeros/inf k={k}")


@pytest.mark.parametrize("k", [1, 20, 64])
def test_shortlist_ties_by_vocab_id(k):
    V = 131_072
    x = synth.levels_block(8, 24, V, [0.0, 2.0, -1.0])
    m = synth.shortlist_map(8, V)
    gu.assert_topk_equal(gu.run_topk(x, k, id_map=m), oracle.topk_mapped(x, k, m), f"mapped ties k={k}")


@pytest.mark.parametrize("gamma", [1, 7, 15])
def test_verify_edges(gamma):
    for V, lanes in ((1, 3), (2, 5), (17, 64), (4099, 33), (248_046, 2)):
        tgt, drafts, acc_p, _ = synth.planted_verify(100 + V, lanes, gamma, V)
        got = gu.run_verify(tgt, drafts, offset=(V + gamma) % 8)
        gu.assert_verify_equal(got, oracle.verify(tgt, drafts), f"planted V={V} gamma={gamma}")
        assert got[0].tolist() == acc_p.tolist()
        # heavy ties and out-of-range drafts
        x = synth.levels_block(200 + V, lanes * (gamma + 1), V, [0.0, 1.0, -0.0])
        d = synth.random_drafts(300 + V, lanes, gamma, V + 3) - 1       # some -1 and >= V
        d[::2] = 0
        gu.assert_verify_equal(gu.run_verify(x, d), oracle.verify(x, d), f"ties V={V} gamma={gamma}")


def test_round_matches_separate_calls_and_repeats():
    """Tickets are reset by the kernel: back-to-back launches on fresh data."""
    for rep in range(3):
        r = synth.make_c2(seed=20 + rep, V=50_000 + 7 * rep)
        v, i, a, c = gu.run_round(r.draft, r.k, r.target, r.drafts, offset=rep)
        gu.assert_topk_equal((v, i), oracle.topk(r.draft, r.k), f"repeat {rep}")
        gu.assert_verify_equal((a, c), oracle.verify(r.target, r.drafts), f"repeat {rep}")


def test_round_counters_accumulate():
    """spec_round_counted: the same outputs as spec_round, and the counter
    block gains exactly the oracle's counts of each round (accumulated over
    rounds of different gamma; NULL counters count nothing)."""
    import torch
    sd = gu.sd_module()
    cnt = sd.new_counters()
    want = {"rounds": 0, "drafted_tokens": 0, "accepted_tokens": 0,
            "position_drafted": [0] * sd.SPEC_MAX_GAMMA, "position_accepted": [0] * sd.SPEC_MAX_GAMMA}
    cases = [synth.make_c2(seed=41, V=40_000), synth.make_c3(seed=42, V=30_001), synth.make_c1(seed=43, V=20_000)]
    for r in cases:
        x, t = gu.dev_u16(r.draft), gu.dev_u16(r.target)
        vals = torch.empty((r.cols, r.k), dtype=torch.int16, device="cuda")
        ids = torch.empty((r.cols, r.k), dtype=torch.int32, device="cuda")
        acc = torch.empty(r.lanes, dtype=torch.int32, device="cuda")
        com = torch.empty((r.lanes, r.gamma + 1), dtype=torch.int32, device="cuda")
        sd.spec_round_counted(x, r.cols, r.V, r.k, vals, ids, t, gu.dev_i32(r.drafts), r.lanes, r.gamma, acc, com,
                              cnt)
        torch.cuda.synchronize()
        sd.spec_device_status()
        wa, wc = oracle.verify(r.target, r.drafts)
        gu.assert_verify_equal((acc.cpu().numpy(), com.cpu().numpy()), (wa, wc), "counted round")
        gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()), oracle.topk(r.draft, r.k),
                             "counted round")
        c = oracle.counters(wa, r.gamma)
        for key in ("rounds", "drafted_tokens", "accepted_tokens"):
            want[key] += c[key]
        for i in range(r.gamma):
            want["position_drafted"][i] += c["position_drafted"][i]
            want["position_accepted"][i] += c["position_accepted"][i]
        assert sd.read_counters(cnt) == want
    # NULL: no counting
    r = cases[0]
    x, t = gu.dev_u16(r.draft), gu.dev_u16(r.target)
    vals = torch.empty((r.cols, r.k), dtype=torch.int16, device="cuda")
    ids = torch.empty((r.cols, r.k), dtype=torch.int32, device="cuda")
    acc = torch.empty(r.lanes, dtype=torch.int32, device="cuda")
    com = torch.empty((r.lanes, r.gamma + 1), dtype=torch.int32, device="cuda")
    sd.spec_round_counted(x, r.cols, r.V, r.k, vals, ids, t, gu.dev_i32(r.drafts), r.lanes, r.gamma, acc, com, None)
    torch.cuda.synchronize()
    assert sd.read_counters(cnt) == want


def _flat_sampled_round(seed: int, lanes: int, gamma: int, V: int):
    """Target columns of plain N(0,1) noise, each draft one of its column's
    five best tokens: acceptance is a real coin flip at every position."""
    from types import SimpleNamespace
    t = synth._draft_block(seed, lanes * (gamma + 1), V, 1.0)
    _, ids = oracle.topk(t, 5)
    pick = synth.rng(seed, 1).integers(0, 5, size=(lanes, gamma))
    drafts = np.array([[ids[l * (gamma + 1) + j, pick[l, j]] for j in range(gamma)] for l in range(lanes)],
                      dtype=np.int32)
    return SimpleNamespace(target=t.reshape(lanes, gamma + 1, V), drafts=drafts, lanes=lanes, gamma=gamma)


@pytest.mark.parametrize("temperature,top_p,top_k", [(1.0, 0.95, 20), (0.7, 0.9, 8), (1.5, 1.0, 64), (2.0, 0.5, 33)])
def test_sampled_verify(temperature, top_p, top_k):
    """spec_verify_sampled against the oracle, bit-exact, on seeded rounds
    whose accept/draw decisions all lie well clear of a boundary (both sides
    compute in float64; exp may differ in the last place)."""
    cases = [(synth.make_c1(seed=51, V=30_000), 0), (synth.make_c2(seed=52, V=20_003), 3),
             (synth.make_c3(seed=53, V=10_001), 5), (_flat_sampled_round(55, 12, 5, 40_000), 1)]
    for i, (r, off) in enumerate(cases):
        u = synth.rng(900 + i, int(top_k)).random((r.lanes, r.gamma + 1, 2))
        wa, wc, margin = oracle.sampled_verify(r.target, r.drafts, temperature, top_p, top_k, u)
        assert margin > 1e-9, margin
        got = gu.run_verify_sampled(r.target, r.drafts, temperature, top_p, top_k, u, offset=off)
        gu.assert_verify_equal(got, (wa, wc), f"sampled T={temperature} top_p={top_p} top_k={top_k} case {i}")


def test_sampled_verify_full_vocabulary():
    """The pages' sampled setting (T 1.0, top_p 0.95, top_k 20) on the C2
    verify part at V = 248,046."""
    r = synth.make_c2()
    u = synth.rng(950, 0).random((r.lanes, r.gamma + 1, 2))
    wa, wc, margin = oracle.sampled_verify(r.target, r.drafts, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal(gu.run_verify_sampled(r.target, r.drafts, 1.0, 0.95, 20, u), (wa, wc), "sampled C2")


def _near_boundary_round(seed, lanes, gamma, V, delta, top_k=20, top_p=0.95):
    """Drafts and uniforms that put every decision `delta` from its boundary:
    draft j is the second token of its column's nucleus; u = q(draft) +/-
    delta (alternating), and where that rejects, u2 puts the draw's target
    delta above or below the running weight after the first kept token."""
    t = synth._draft_block(seed, lanes * (gamma + 1), V, 3.0)
    vals, ids = oracle.topk(t, top_k)
    drafts = np.empty((lanes, gamma), dtype=np.int32)
    u = np.empty((lanes, gamma + 1, 2))
    g = synth.rng(seed + 1, 0)
    for ln in range(lanes):
        for j in range(gamma + 1):
            kept, q = oracle.sampled_column(vals[ln * (gamma + 1) + j], ids[ln * (gamma + 1) + j], 1.0, top_p)
            sign = 1.0 if (ln + j) % 2 else -1.0
            if j < gamma:
                d = kept[1] if len(kept) > 1 else kept[0]
                drafts[ln, j] = d
                u[ln, j, 0] = min(max(q[kept.index(d)] + sign * delta, 0.0), 1.0 - 1e-12)
            else:
                d = None
                u[ln, j, 0] = g.random()
            w = [qt for tok, qt in zip(kept, q) if tok != d]
            W = float(np.sum(np.array(w, dtype=np.float64))) if w else 1.0
            r1 = w[0] if w else 0.5
            u[ln, j, 1] = min(max((r1 - sign * delta) / W, 0.0), 1.0 - 1e-12)
    return t, drafts, u


@pytest.mark.parametrize("delta", [5e-5, 3e-6])
def test_sampled_decisions_near_boundaries(delta):
    """Every acceptance and draw lies `delta` from its boundary -- inside the
    float32 path's margin, so the kernels decide these in float64 -- and
    must agree with the oracle."""
    lanes, gamma, V = 6, 7, 50_021
    t, drafts, u = _near_boundary_round(970 + int(delta * 1e7), lanes, gamma, V, delta)
    wa, wc, margin = oracle.sampled_verify(t, drafts, 1.0, 0.95, 20, u)
    assert 1e-9 < margin <= delta * 1.01
    gu.assert_verify_equal(gu.run_verify_sampled(t.reshape(lanes, gamma + 1, V), drafts, 1.0, 0.95, 20, u),
                           (wa, wc), f"sampled near boundaries delta={delta}")


@pytest.mark.parametrize("V", [248_046, 131_072])
def test_sampled_verify_many_columns(V):
    """Sampled verify over 40 lanes x 8 target columns: enough columns for
    the group-maxima kernel's finishing warps (12 + 4 warps at the full
    vocabulary; 8 + 8 for top_k 20 on shortlist-length columns)."""
    lanes, gamma = 40, 7
    t = synth._draft_block(990 + V % 97, lanes * (gamma + 1), V, 3.0)
    _, top = oracle.topk(t, 1)   # drafts: each position's most likely token, so some are accepted
    drafts = np.ascontiguousarray(top[:, 0].reshape(lanes, gamma + 1)[:, :gamma], dtype=np.int32)
    u = synth.rng(992, 0).random((lanes, gamma + 1, 2))
    wa, wc, margin = oracle.sampled_verify(t, drafts, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal(gu.run_verify_sampled(t.reshape(lanes, gamma + 1, V), drafts, 1.0, 0.95, 20, u),
                           (wa, wc), f"sampled many columns V={V}")


def test_round_sampled_is_topk_plus_sampled_verify():
    import torch
    sd = gu.sd_module()
    r = synth.make_c2(seed=56, V=30_011)
    u = synth.rng(970, 0).random((r.lanes, r.gamma + 1, 2))
    x, t = gu.dev_u16(r.draft), gu.dev_u16(r.target, 2)
    vals = torch.empty((r.cols, r.k), dtype=torch.int16, device="cuda")
    ids = torch.empty((r.cols, r.k), dtype=torch.int32, device="cuda")
    acc = torch.empty(r.lanes, dtype=torch.int32, device="cuda")
    com = torch.empty((r.lanes, r.gamma + 1), dtype=torch.int32, device="cuda")
    ut = torch.from_numpy(u).cuda()
    sd.spec_round_sampled(x, r.cols, r.V, r.k, vals, ids, t, gu.dev_i32(r.drafts), r.lanes, r.gamma, 1.0, 0.95, 20,
                          ut, acc, com)
    torch.cuda.synchronize()
    sd.spec_device_status()
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()), oracle.topk(r.draft, r.k),
                         "round_sampled top-k")
    wa, wc, margin = oracle.sampled_verify(r.target, r.drafts, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal((acc.cpu().numpy(), com.cpu().numpy()), (wa, wc), "round_sampled verify")


def test_sampled_verify_small_and_tied():
    """Tiny vocabularies (top_k = V), all-tied columns (a uniform q: every
    draw walks the id order) and ragged phases."""
    for V, gamma, lanes in ((1, 1, 3), (2, 3, 5), (5, 4, 7), (17, 15, 2)):
        t = synth._draft_block(70 + V, lanes * (gamma + 1), V, 1.0)
        t[::3] = synth.bf16_bits(0.5)                           # every third column all tied
        drafts = synth.rng(71 + V, 0).integers(-1, V + 1, size=(lanes, gamma)).astype(np.int32)
        u = synth.rng(72 + V, 0).random((lanes, gamma + 1, 2))
        for top_k, top_p in ((V, 1.0), (max(1, V // 2), 0.8), (1, 0.95)):
            wa, wc, margin = oracle.sampled_verify(t, drafts, 1.0, top_p, top_k, u)
            if margin <= 1e-9:
                continue   # a decision on a boundary: float64 exp may round either way
            got = gu.run_verify_sampled(t.reshape(lanes, gamma + 1, V), drafts, 1.0, top_p, top_k, u,
                                        offset=(V + gamma) % 8)
            gu.assert_verify_equal(got, (wa, wc), f"sampled V={V} gamma={gamma} top_k={top_k} top_p={top_p}")


def test_sampled_top_k_one_is_greedy():
    r = synth.make_c3(seed=54, V=7_777)
    u = synth.rng(960, 0).random((r.lanes, r.gamma + 1, 2))
    gu.assert_verify_equal(gu.run_verify_sampled(r.target, r.drafts, 0.8, 0.95, 1, u),
                           oracle.verify(r.target, r.drafts), "sampled top_k=1")


@pytest.mark.parametrize("k", [1, 8, 64])
def test_column_over_many_units(k):
    """One column of a million logits: about 120 CTAs (or 240 warps) share
    it, so the completing unit merges lists more than 32 at a time."""
    V = 1_000_000
    x = synth._draft_block(80 + k, 1, V, 3.0)
    gu.assert_topk_equal(gu.run_topk(x, k, offset=3), oracle.topk(x, k), f"one column V={V} k={k}")


@pytest.mark.parametrize("k", [8, 64])
def test_rounds_of_a_million_vectors(k):
    """24 draft columns and a lane of 8 target columns at V = 248,046 (about
    a million 16-byte vectors: more than 4,096 a CTA on a full grid, so the
    group-maxima kernel's one-pass mode holds 16 vectors a thread), and a
    sampled verify of 4 such lanes alone."""
    V = synth.VOCAB
    x = synth._draft_block(95 + k, 24, V, 3.0)
    tgt, drafts, _, _ = synth.planted_verify(96 + k, 1, 7, V)
    v, i, a, c = gu.run_round(x, k, tgt, drafts, offset=k % 8)
    gu.assert_topk_equal((v, i), oracle.topk(x, k), f"24 columns k={k}")
    gu.assert_verify_equal((a, c), oracle.verify(tgt, drafts), f"24 columns k={k} verify")
    t4, d4, _, _ = synth.planted_verify(97 + k, 4, 7, V)
    u = synth.rng(98 + k, 0).random((4, 8, 2))
    wa, wc, margin = oracle.sampled_verify(t4, d4, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal(gu.run_verify_sampled(t4, d4, 1.0, 0.95, 20, u), (wa, wc), "sampled 4 lanes")


@pytest.mark.parametrize("cols,k", [(60, 20), (40, 64), (40, 1)])
def test_columns_in_clusters(cols, k):
    """Rounds with fewer columns than three quarters of the SMs and too many
    vectors for one pass, which the group-maxima kernel runs as whole columns
    in thread-block clusters (2 or 3 CTAs a column): three-level ties and
    noise columns, the top-k of each."""
    V = synth.VOCAB
    x = synth.levels_block(70 + cols + k, cols, V, [0.0, 1.0, -0.0])
    x[1::2] = synth._draft_block(71 + cols + k, cols // 2, V, 3.0)
    gu.assert_topk_equal(gu.run_topk(x, k, offset=k % 8), oracle.topk(x, k), f"{cols} columns k={k}")


def test_verify_in_clusters():
    """Greedy and sampled verify of 5 lanes of 8 columns at V = 248,046 (40
    columns: three CTAs a column in a cluster), half the lanes accepting
    every draft."""
    V, lanes, gamma = synth.VOCAB, 5, 7
    t, d, _, _ = synth.planted_verify(80, lanes, gamma, V)
    gu.assert_verify_equal(gu.run_verify(t, d), oracle.verify(t, d), "greedy, 40 columns")
    u = synth.rng(81, 0).random((lanes, gamma + 1, 2))
    wa, wc, margin = oracle.sampled_verify(t, d, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal(gu.run_verify_sampled(t, d, 1.0, 0.95, 20, u), (wa, wc), "sampled, 40 columns")


def test_verify_columns_over_many_units():
    """A lane of four target columns of a million logits each (greedy and
    sampled): every column is shared by dozens of units."""
    V, gamma = 1_000_000, 3
    t = synth._draft_block(90, gamma + 1, V, 1.0)
    _, ids = oracle.topk(t, 3)
    drafts = np.array([[ids[0, 0], ids[1, 0], ids[2, 1]]], dtype=np.int32)
    gu.assert_verify_equal(gu.run_verify(t.reshape(1, gamma + 1, V), drafts), oracle.verify(t, drafts),
                           "verify V=1e6")
    u = synth.rng(91, 0).random((1, gamma + 1, 2))
    wa, wc, margin = oracle.sampled_verify(t, drafts, 1.0, 0.95, 20, u)
    assert margin > 1e-9
    gu.assert_verify_equal(gu.run_verify_sampled(t.reshape(1, gamma + 1, V), drafts, 1.0, 0.95, 20, u),
                           (wa, wc), "sampled V=1e6")


def test_empty_and_rejected_calls_write_nothing():
    import torch
    sd = gu.sd_module()
    x = gu.dev_u16(np.zeros((3, 100), dtype=np.uint16))
    vals = gu.Guarded(3 * 8, torch.int16)
    ids = gu.Guarded(3 * 8, torch.int32)
    sd.spec_topk(x, 0, 100, 8, vals.view, ids.view)
    with pytest.raises(sd.SpecError):
        sd.spec_topk(x, 3, 100, 101, vals.view, ids.view)
    torch.cuda.synchronize()
    for g in (vals, ids):
        g.check_guards()
        assert np.all(g.host() == g.sent)


def test_side_stream_and_graph_capture():
    import torch
    sd = gu.sd_module()
    r = synth.make_c1(seed=4, V=100_003)
    r2 = synth.make_c1(seed=5, V=100_003)
    x = gu.dev_u16(r.draft)
    t = gu.dev_u16(r.target)
    d = gu.dev_i32(r.drafts)
    cols, V, k, lanes, gamma = r.cols, r.V, r.k, r.lanes, r.gamma
    vals = torch.empty((cols, k), dtype=torch.int16, device="cuda")
    ids = torch.empty((cols, k), dtype=torch.int32, device="cuda")
    acc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    com = torch.empty((lanes, gamma + 1), dtype=torch.int32, device="cuda")
    sd.spec_reserve(cols, k, lanes, gamma)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sd.spec_round(x, cols, V, k, vals, ids, t, d, lanes, gamma, acc, com)
    s.synchronize()
    gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()), oracle.topk(r.draft, k), "stream")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sd.spec_round(x, cols, V, k, vals, ids, t, d, lanes, gamma, acc, com)
    for rr in (r2, r, r2):
        x.copy_(torch.from_numpy(rr.draft.view(np.int16)))
        t.copy_(torch.from_numpy(rr.target.view(np.int16)))
        d.copy_(torch.from_numpy(rr.drafts))
        g.replay()
        torch.cuda.synchronize()
        gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()), oracle.topk(rr.draft, k),
                             "graph replay")
        gu.assert_verify_equal((acc.cpu().numpy(), com.cpu().numpy()), oracle.verify(rr.target, rr.drafts),
                               "graph replay verify")
    sd.spec_set_stream(None)


def test_graph_survives_scratch_growth():
    """A graph captured before the scratch grows replays correctly after it:
    the area it captured stays allocated (retired, not freed) while a larger
    one serves new calls."""
    import torch
    sd = gu.sd_module()
    r = synth.make_c1(seed=6, V=50_001)
    x, t, d = gu.dev_u16(r.draft), gu.dev_u16(r.target), gu.dev_i32(r.drafts)
    cols, V, k, lanes, gamma = r.cols, r.V, r.k, r.lanes, r.gamma
    vals = torch.empty((cols, k), dtype=torch.int16, device="cuda")
    ids = torch.empty((cols, k), dtype=torch.int32, device="cuda")
    acc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    com = torch.empty((lanes, gamma + 1), dtype=torch.int32, device="cuda")
    sd.spec_reserve(cols, k, lanes, gamma)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sd.spec_round(x, cols, V, k, vals, ids, t, d, lanes, gamma, acc, com)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sd.spec_round(x, cols, V, k, vals, ids, t, d, lanes, gamma, acc, com)
    sd.spec_set_stream(None)
    # larger than any round of the suite: every region moves to a new area
    sd.spec_reserve(3_000_000, 64, 8192, 15)
    big = synth.make_c2(seed=7, V=20_011)
    got = gu.run_round(big.draft, big.k, big.target, big.drafts)
    gu.assert_topk_equal(got[:2], oracle.topk(big.draft, big.k), "after growth")
    gu.assert_verify_equal(got[2:], oracle.verify(big.target, big.drafts), "after growth verify")
    torch.cuda.synchronize()
    for _ in range(2):
        with torch.cuda.stream(s):
            vals.zero_()
            acc.fill_(-7)
            g.replay()
        s.synchronize()
        sd.spec_device_status()
        gu.assert_topk_equal((vals.cpu().numpy().view(np.uint16), ids.cpu().numpy()), oracle.topk(r.draft, k),
                             "old graph after growth")
        gu.assert_verify_equal((acc.cpu().numpy(), com.cpu().numpy()), oracle.verify(r.target, r.drafts),
                               "old graph after growth verify")
    del g
    sd.spec_release()


def test_round_host_buffers():
    sd = gu.sd_module()
    r = synth.make_c2(seed=9, V=30_000)
    vals = np.zeros((r.cols, r.k), dtype=np.uint16)
    ids = np.zeros((r.cols, r.k), dtype=np.int32)
    acc = np.zeros(r.lanes, dtype=np.int32)
    com = np.zeros((r.lanes, r.gamma + 1), dtype=np.int32)
    sd.spec_round_host(r.draft, r.cols, r.V, r.k, vals, ids, r.target, r.drafts, r.lanes, r.gamma, acc, com)
    gu.assert_topk_equal((vals, ids), oracle.topk(r.draft, r.k), "host buffers")
    gu.assert_verify_equal((acc, com), oracle.verify(r.target, r.drafts), "host buffers")


def test_bounded_wait_gives_up_and_is_reported(kernel):
    """Failure detection without a fault: a wait on a barrier nothing
    arrives on gives up after its limit, the device flag is reported once
    by spec_device_status, and the CTA's next wait returns at once."""
    import torch
    sd = gu.sd_module()
    sd.spec_device_status()                        # nothing pending
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    sd._check(sd.lib.spec_selftest_wait_timeout(2_000_000, out.data_ptr()))   # 2 ms
    torch.cuda.synchronize()
    first_ok, first_ns, second_ok, second_ns = (int(v) for v in out.cpu())
    assert first_ok == 0 and first_ns >= 2_000_000
    assert second_ok == 0 and second_ns < 1_000_000
    with pytest.raises(sd.SpecError) as ei:
        sd.spec_device_status()
    assert "gave up a bounded wait" in str(ei.value)
    sd.spec_device_status()                        # cleared by the report
