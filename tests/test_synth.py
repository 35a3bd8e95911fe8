"""The seeded input generator: published SplitMix64 vectors, bf16 rounding, value statistics."""
import numpy as np

import synth
from synth import workloads as W


def test_splitmix64_published_stream_seed0():
    # SplitMix64 (Steele, Lea & Flood 2014) seeded with 0: the first three outputs
    s = np.array([0, 1, 2], dtype=np.uint64) * synth.GOLDEN
    out = synth.mix64(s)
    assert [hex(int(x)) for x in out] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4",
                                          "0x6c45d188009454f"]


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 1.0 + 2**-8 + 2**-20, 3.0],
                 dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0, 1.0 + 4 * 2**-8, -1.0,
                                                 1.0 + 2**-7, 3.0], dtype=np.float32))


def test_values_are_standardised_and_bounded():
    h = synth.prefix_hashes(7, synth.tokens(7, 1, 4000))
    v = synth.values_f32(h, synth.TENSOR_K, 3, range(4), 128)
    assert abs(float(v.mean())) < 0.01
    assert abs(float(v.var()) - 1.0) < 0.01
    assert np.abs(v).max() <= np.sqrt(3.0) * 2 + 1e-6
    # the values are a function of (prefix hash, tensor, layer, head) only
    v2 = synth.values_f32(h[::-1], synth.TENSOR_K, 3, [2], 128)
    np.testing.assert_array_equal(v2[::-1, 0], v[:, 2])
    assert not np.array_equal(synth.values_f32(h[:5], synth.TENSOR_V, 3, [0], 128),
                              v[:5, :1])


def test_prefix_hash_depends_only_on_prefix():
    a = np.array([5, 6, 7, 8], dtype=np.int32)
    b = np.array([5, 6, 9, 8], dtype=np.int32)
    ha, hb = synth.prefix_hashes(0, a), synth.prefix_hashes(0, b)
    assert ha[0] == hb[0] and ha[1] == hb[1] and ha[2] != hb[2] and ha[3] != hb[3]
    hab = synth.prefix_hashes_batch(0, [a, b, a[:2]])
    np.testing.assert_array_equal(hab[0], ha)
    np.testing.assert_array_equal(hab[1], hb)
    np.testing.assert_array_equal(hab[2], ha[:2])


def test_permutation_is_a_permutation():
    p = synth.permutation(3, 1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not np.array_equal(p, np.arange(1000))


def test_workload_shapes():
    w = W.tiny_extend()
    assert [len(s) for s in w.phases[0].seqs + w.phases[1].seqs] == [80] * 4
    firsts = {int(s[64]) for s in w.phases[0].seqs + w.phases[1].seqs}
    assert len(firsts) == 4
    w = W.few_shot_extend()
    assert len(w.phases[1].seqs) == 64 and all(len(s) == 2050 for s in w.phases[1].seqs)
    w = W.two_level_extend()
    assert len(w.phases[2].seqs) == 64 and all(len(s) == 1120 for s in w.phases[2].seqs)
    L = W.decode_lengths_lognormal(0, 256)
    assert L.min() >= 128 and L.max() <= 16384 and 1500 < np.median(L) < 2800
