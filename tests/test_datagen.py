"""The seeded input generator: determinism, sub-range regeneration, distributions."""
import numpy as np

import datagen


def test_counter_based_subrange():
    full = datagen.u8(7, 1000)
    assert np.array_equal(full[123:456], datagen.u8(7, 333, start=123))
    nf = datagen.normal_f32(9, 999)
    assert np.array_equal(nf[101:700], datagen.normal_f32(9, 599, start=101))


def test_streams_and_seeds_differ():
    assert not np.array_equal(datagen.u8(1, 64), datagen.u8(2, 64))
    assert not np.array_equal(datagen.u8(1, 64, seed=0), datagen.u8(1, 64, seed=1))


def test_distributions():
    b = datagen.u8(3, 1 << 20)
    counts = np.bincount(b, minlength=256)
    assert counts.min() > 3600 and counts.max() < 4600
    z = datagen.normal_f32(4, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    i8 = datagen.int8_sym(5, 1 << 18, 127)
    assert i8.min() == -127 and i8.max() == 127
    s = datagen.absnormal_f32(6, 1 << 16, 0.02, 1e-4)
    assert s.min() >= np.float32(1e-4) and abs(s.mean() - (0.02 * np.sqrt(2 / np.pi) + 1e-4)) < 5e-4
    bf = datagen.bf16_bits_to_f32(datagen.normal_bf16_bits(4, 1000))
    ref = datagen.normal_f32(4, 1000)
    assert np.all(np.abs(bf - ref) <= np.abs(ref) * 2.0 ** -8)


def test_choose_distinct():
    c = datagen.choose(16, 160, 16)
    assert len(set(c.tolist())) == 16 and c.min() >= 0 and c.max() < 160


def test_moe_weights_subset_matches_full():
    full = datagen.moe_weights(6, 128, 64)
    sub = datagen.moe_weights(6, 128, 64, experts=[4, 1])
    for key in full:
        assert np.array_equal(sub[key][0], full[key][4])
        assert np.array_equal(sub[key][1], full[key][1])


def test_moe_inputs_token_subrange():
    x, l = datagen.moe_inputs(8, 160, 256, hot=16)
    x2, l2 = datagen.moe_inputs(3, 160, 256, hot=16, token_start=5)
    assert np.array_equal(x[5:], x2) and np.array_equal(l[5:], l2)
    hot = datagen.hot_experts(160, 16)
    # the hot experts are boosted: they take most of the top-8 picks
    top = np.argsort(-l, axis=1)[:, :8]
    assert np.isin(top, hot).mean() > 0.5
