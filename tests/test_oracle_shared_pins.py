"""Pins of the oracle's shared-expert path ("kimi-k3-mlx", Architecture table: always-on shared
experts on the residual, beside the routed ones) against facts that do not come from the oracle:
a hand-worked one-hot case, exact invariants (zero weights, power-of-two scaling, expert order)
and float64 library matrix products on the tiny configuration. Runs without a GPU."""
import math

import numpy as np

import oracle
import synth

NS, IS = 2, 64  # two shared experts of width 64 on the tiny configuration


def _nearest_bf16(x):
    """Round-to-nearest-even to 8 significant bits (normal range), stated independently."""
    if x == 0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)
    return round(m * 256) * math.ldexp(1.0, e - 8)


def _bf16_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0] >> 16)


def _layer(shared, seed=0, zero_out=False):
    d = synth.TINY
    wr, wi, wo = synth.host_dense(d, seed)
    if zero_out:
        wo = np.zeros_like(wo)
    ex = {e: synth.host_expert(d, seed, e) for e in range(d.n_experts)}
    return oracle.Layer(d, wr, wi, wo, ex, shared=shared)


def test_shared_one_hot_closed_form():
    d = synth.TINY
    H, S = d.hidden, NS * IS
    g = np.zeros((S, H), np.uint16)
    u = np.zeros((S, H), np.uint16)
    dn = np.zeros((H, S), np.uint16)
    r, h0, h1, ho = IS + 3, 11, 40, 7          # expert 1, its row 3; inputs h0, h1; output ho
    g[r, h0] = _bf16_bits(2.0)
    u[r, h1] = _bf16_bits(0.5)
    dn[ho, r] = _bf16_bits(-1.0)
    lay = _layer((g, u, dn, NS))
    x = synth.host_bf16_normal(3, synth.S_X, 0, H, 1.0)
    s, a = lay.shared_ffn(x)
    xf = oracle.bf16_to_f64(x)
    gv, uv = 2.0 * xf[h0], 0.5 * xf[h1]
    a_r = _nearest_bf16(gv / (1.0 + math.exp(-gv)) * uv)  # the gate half is the activated one
    want = np.zeros(H)
    want[ho] = -a_r
    np.testing.assert_array_equal(s, want)
    assert oracle.bf16_to_f64(a)[r] == a_r and np.count_nonzero(oracle.bf16_to_f64(a)) <= 1


def test_shared_zero_weights_leave_the_layer_bit_identical():
    d = synth.TINY
    H, S = d.hidden, NS * IS
    z = np.zeros((S, H), np.uint16)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y0 = _layer(None).forward(x)["y"]
    y1 = _layer((z, z, np.zeros((H, S), np.uint16), NS)).forward(x)["y"]
    np.testing.assert_array_equal(y1, y0)


def test_shared_down_times_two_doubles_y_exactly():
    """With W_out = 0, y = bf16(s); doubling every down weight doubles s and y exactly."""
    d = synth.TINY
    g, u, dn = synth.host_shared(d, NS, IS, 5)
    dn2 = (oracle.bf16_to_f64(dn) * 2).astype(np.float32).view(np.uint32) >> 16
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y1 = oracle.bf16_to_f64(_layer((g, u, dn, NS), zero_out=True).forward(x)["y"])
    y2 = oracle.bf16_to_f64(_layer((g, u, dn2.astype(np.uint16), NS), zero_out=True).forward(x)["y"])
    assert np.count_nonzero(y1) > 0.9 * y1.size
    np.testing.assert_array_equal(y2, 2 * y1)


def test_shared_expert_order_does_not_matter():
    d = synth.TINY
    g, u, dn = synth.host_shared(d, NS, IS, 6)
    sw = np.r_[IS:2 * IS, 0:IS]
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y1 = _layer((g, u, dn, NS)).forward(x)["y"]
    y2 = _layer((g[sw], u[sw], dn[:, sw], NS)).forward(x)["y"]
    np.testing.assert_array_equal(y2, y1)


def test_shared_vs_numpy_matmuls():
    """s = D bf16(silu(G x) * (U x)) as float64 library products; y = bf16(W_out c + s)."""
    d = synth.TINY
    g, u, dn = synth.host_shared(d, NS, IS, 7)
    lay = _layer((g, u, dn, NS), zero_out=True)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    xf = oracle.bf16_to_f64(x)
    gv = xf @ oracle.bf16_to_f64(g).T
    uv = xf @ oracle.bf16_to_f64(u).T
    a = np.vectorize(_nearest_bf16)(gv / (1.0 + np.exp(-gv)) * uv)
    s = a @ oracle.bf16_to_f64(dn).T
    for t in range(x.shape[0]):
        so, ao = lay.shared_ffn(x[t])
        np.testing.assert_array_equal(oracle.bf16_to_f64(ao), a[t])  # same roundings, exact inputs
        np.testing.assert_allclose(so, s[t], rtol=1e-12, atol=1e-12)
    y = oracle.bf16_to_f64(lay.forward(x)["y"])
    want = np.vectorize(_nearest_bf16)(s)
    assert np.mean(y == want) > 0.999  # summation order can move a value across a rounding tie
    np.testing.assert_allclose(y, want, rtol=2.0**-8)


def test_shared_and_routed_add_before_rounding():
    """Both parts present: y = bf16(W_out c + s), one rounding of the exact sum."""
    d = synth.TINY
    g, u, dn = synth.host_shared(d, NS, IS, 8)
    lay = _layer((g, u, dn, NS))
    x = synth.host_x(synth.WORKLOADS["tiny"])
    r = lay.forward(x)
    wo = oracle.bf16_to_f64(synth.host_dense(d, 0)[2])
    for t in range(x.shape[0]):
        s, _ = lay.shared_ffn(x[t])
        yo = oracle.bf16_to_f64(r["c"][t]) @ wo.T + s
        got = oracle.bf16_to_f64(r["y"][t])
        assert np.mean(got == np.vectorize(_nearest_bf16)(yo)) > 0.99
