"""Pins of the oracle's MXFP4 activation mode (actq = 2: e2m1 elements with one e8m0 exponent
per 32, the 4-bit activations the fp4 tensor rate needs; the hot-path table's next row; the
library does not run it yet). The rule is the OCP Microscaling (MX) v1.0 conversion for FP4:
shared exponent floor(log2 amax) - 2 (E2M1's largest exponent), elements rounded to nearest
with ties to even, saturating at 6. Pinned by hand-worked cases, exact round trips, power-of-two
scaling, an independent statement of the rule, and a tiny layer against numpy."""
import math

import numpy as np
import pytest

import oracle
import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # magnitudes of codes 0..7 (OCP MX v1.0)


def _e2m1_round(x):
    """Independent: nearest e2m1 magnitude, ties to the even code, saturating at 6."""
    a = abs(x)
    if a >= 6.0:
        q = 6.0
    else:
        best = min(range(8), key=lambda c: (abs(a - E2M1[c]), c & 1))
        q = E2M1[best]
    return -q if math.copysign(1.0, x) < 0 else q


def _mxfp4_block(v):
    amax = max(abs(x) for x in v)
    if amax == 0.0:
        return [0.0] * 32
    X = max(-127, min(127, math.floor(math.log2(amax)) - 2))
    return [_e2m1_round(x / 2.0 ** X) * 2.0 ** X for x in v]


@pytest.mark.parametrize("x,want", [
    (0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0), (5.0, 4.0),
    (5.5, 6.0), (6.0, 6.0), (7.9, 6.0), (100.0, 6.0), (0.3, 0.5), (-2.5, -2.0), (-5.0, -4.0),
    (-9.0, -6.0), (0.0, 0.0)])
def test_e2m1_rounding_hand_worked(x, want):
    """Midpoints go to the even code (0, 1.0, 2.0, 4.0 are codes 0, 2, 4, 6); beyond 6 saturates."""
    code = oracle.e2m1_encode(x)
    assert oracle.e2m1(code) == want
    if x < 0:
        assert code & 8


def test_representable_blocks_round_trip_exactly():
    rng = np.random.default_rng(3)
    for X in (-20, -3, 0, 5, 30):
        mags = rng.choice(E2M1, 32)
        mags[0] = 6.0 if X % 2 else 4.0  # fix amax so the shared exponent is X exactly
        v = mags * rng.choice([-1.0, 1.0], 32) * 2.0 ** X
        np.testing.assert_array_equal(oracle.mxfp4_roundtrip(v), v)
        codes, sc = oracle.mxfp4_block(v)
        assert sc == X + 127


def test_power_of_two_scaling_moves_only_the_exponent():
    rng = np.random.default_rng(4)
    v = rng.normal(0, 1.0, 32)
    c0, s0 = oracle.mxfp4_block(v)
    for m in (-7, 1, 9):
        c1, s1 = oracle.mxfp4_block(v * 2.0 ** m)
        np.testing.assert_array_equal(c1, c0)
        assert s1 == s0 + m


def test_block_rule_vs_independent_statement():
    rng = np.random.default_rng(5)
    for i in range(300):
        v = rng.normal(0, 10.0 ** rng.uniform(-3, 3), 32)
        if i % 7 == 0:
            v[rng.integers(32)] = 0.0
        np.testing.assert_array_equal(oracle.mxfp4_roundtrip(v), _mxfp4_block(list(v)))
    np.testing.assert_array_equal(oracle.mxfp4_roundtrip(np.zeros(32)), np.zeros(32))


def _nearest_bf16(x):
    if x == 0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)
    return round(m * 256) * math.ldexp(1.0, e - 8)


def test_tiny_layer_in_mxfp4_mode_vs_numpy():
    """z and the GLU output a go through the MXFP4 round trip before each expert matrix."""
    d = synth.TINY
    wr, wi, wo = synth.host_dense(d, 0)
    ex = {e: synth.host_expert(d, 0, e) for e in range(d.n_experts)}
    lay = oracle.Layer(d, wr, wi, wo, ex, actq=2)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    r = lay.forward(x)
    xf = oracle.bf16_to_f64(x)
    nb = np.vectorize(_nearest_bf16)
    z = nb(xf @ oracle.bf16_to_f64(wi).T)

    def deq(q, s):
        codes = np.empty((q.shape[0], 2 * q.shape[1]), np.int64)
        codes[:, 0::2], codes[:, 1::2] = q & 0xF, q >> 4
        table = np.array(E2M1 + [-m for m in E2M1])
        return table[codes] * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)

    def rt(vec):
        return np.concatenate([_mxfp4_block(list(vec[b:b + 32])) for b in range(0, len(vec), 32)])

    T, k = x.shape[0], d.top_k
    for t in range(T):
        c = np.zeros(d.latent)
        zq = rt(z[t])
        for j in range(k):
            e = int(r["idx"][t, j])
            G, U, D = (deq(ex[e][a], ex[e][b]) for a, b in (("gate_q", "gate_s"), ("up_q", "up_s"),
                                                             ("down_q", "down_s")))
            g, u = G @ zq, U @ zq
            a = rt(nb(g / (1.0 + np.exp(-g)) * u))
            c += r["w"][t, j] * (D @ a)
        y = nb(oracle.bf16_to_f64(oracle.bf16_from_f64(nb(c))) @ oracle.bf16_to_f64(wo).T)
        got = oracle.bf16_to_f64(r["y"][t])
        assert np.linalg.norm(got - y) <= 1e-6 * np.linalg.norm(y)
