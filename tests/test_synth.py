"""The seeded input generator: reproducible, planted structure realised (no GPU)."""
import numpy as np

import synth


def test_reproducible_and_chunk_independent():
    a = synth._draft_block(9, 5, 1001, 3.0)
    b = synth._draft_block(9, 3, 1001, 3.0)
    assert np.array_equal(a[:3], b)
    assert synth.content_hash(a) == synth.content_hash(synth._draft_block(9, 5, 1001, 3.0))
    assert synth.content_hash(a) != synth.content_hash(synth._draft_block(10, 5, 1001, 3.0))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, -0.0, 3.0e38], dtype=np.float32)
    b = synth.f32_to_bf16_bits(x)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert b[0] == 0x3F80 and b[1] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    assert b[2] == 0x3F82
    assert b[3] == 0xC020 and b[4] == 0x0000 and b[5] == 0x8000
    back = synth.bf16_to_f32(b)
    assert np.all(np.abs(back[:4] - x[:4]) <= 2 ** -8 * np.abs(x[:4]))


def test_no_nan_and_noise_below_peaks():
    x = synth._draft_block(2, 4, 50_000, 3.0)
    assert not np.any(((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0))
    assert synth.bf16_to_f32(x).max() <= synth.NOISE_CLIP


def test_quantised_levels():
    x = synth._draft_block(3, 2, 40_000, 3.0, quant=True)
    lv = np.unique(synth.bf16_to_f32(x))
    assert len(lv) <= 64 and lv.min() >= -8.0 and lv.max() <= 7.75
    assert np.all(np.asarray(lv * 4) == np.rint(lv * 4))


def test_planted_drafts_small_v():
    for V in (1, 2, 9):
        tgt, drafts, acc, t_arg = synth.planted_verify(5, 6, 4, V, accept=np.array([0, 1, 2, 3, 4, 0]))
        for l in range(6):
            a = int(acc[l])
            assert drafts[l, :a].tolist() == t_arg[l, :a].tolist()
            if a < 4:
                assert drafts[l, a] != t_arg[l, a]


def test_shortlist_map_injective():
    m = synth.shortlist_map(6, 131_072)
    assert m.shape == (131_072,) and len(np.unique(m)) == 131_072
    assert m.min() >= 0 and m.max() < synth.VOCAB


def test_config_shapes_small():
    r = synth.make_c1(V=2_000)
    assert r.draft.shape == (7, 2_000) and r.target.shape == (8, 2_000) and r.drafts.shape == (1, 7)
    assert r.planted_accept.tolist() == [4]
    r3 = synth.make_c3(V=3_000)
    assert r3.target.shape == (48, 3_000) and r3.planted_accept[0] == 15 and r3.planted_accept[1] == 0
