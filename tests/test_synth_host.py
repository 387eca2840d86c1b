"""The shared seeded input generator (host side): determinism, random access and the
distributions the workloads ask for (bf16 ~N(0,1) / ~N(0,0.02), codes U{0..15},
e8m0 U{120..127}, Zipf-skewed expert popularity)."""
import numpy as np

import oracle
import synth


def test_random_access_matches_sequential():
    a = synth.host_bf16_normal(3, 5, 0, 1000, 0.02)
    b = synth.host_bf16_normal(3, 5, 400, 600, 0.02)
    np.testing.assert_array_equal(a[400:], b)
    c = synth.host_bytes(3, 5, 0, 777)
    d = synth.host_bytes(3, 5, 13, 700)
    np.testing.assert_array_equal(c[13:713], d)


def test_distributions():
    x = oracle.bf16_to_f64(synth.host_bf16_normal(0, synth.S_X, 0, 200000, 1.0))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = oracle.bf16_to_f64(synth.host_bf16_normal(0, synth.S_W_IN, 0, 200000, 0.02))
    assert abs(w.std() - 0.02) < 0.0005
    q = synth.host_bytes(0, synth.S_GATE_Q, 0, 200000)
    nib = np.concatenate([q & 0xF, q >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * len(nib) / 16
    s = synth.host_uniform_u8(0, synth.S_GATE_S, 0, 100000, 120, 127)
    assert s.min() == 120 and s.max() == 127
    assert np.bincount(s - 120).min() > 0.9 * 100000 / 8


def test_streams_and_seeds_are_independent():
    a = synth.host_bytes(0, 1, 0, 64)
    assert not np.array_equal(a, synth.host_bytes(0, 2, 0, 64))
    assert not np.array_equal(a, synth.host_bytes(1, 1, 0, 64))


def test_zipf_bias_is_a_permuted_log_rank():
    b = synth.zipf_bias(896, 0)
    ranks = np.exp(-b.astype(np.float64) / 1.1)
    np.testing.assert_allclose(np.sort(ranks), np.arange(1, 897), rtol=1e-5)


def test_topk_sets_are_distinct_and_sorted():
    for skew in ("uniform", "zipf", "one"):
        idx = synth.host_topk_sets(1, 50, 40, 6, skew)
        assert np.all(np.diff(idx, axis=1) > 0)
        assert idx.min() >= 0 and idx.max() < 40
