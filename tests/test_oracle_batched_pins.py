"""Pins of the oracle's batched statement (numpy float64 matrix products, experts decoded once
each; used for parity checks over thousands of tokens) against the scalar C statement and
against independent rules. Runs without a GPU."""
import math

import numpy as np
import pytest

import oracle
import synth


def _nearest_bf16(x: float) -> float:
    """Round to 8 significant bits, ties to even, by Python's exact round() on the mantissa."""
    if x == 0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)
    if e - 1 < -126:  # subnormal bf16: fixed quantum 2^-133
        return round(x / 2.0**-133) * 2.0**-133
    r = round(m * 256) * math.ldexp(1.0, e - 8)
    return math.inf * (1 if r > 0 else -1) if abs(r) >= 2.0**128 else r


def test_bf16_rounding_of_arrays_matches_the_scalar_rule():
    rng = np.random.default_rng(3)
    ties = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 2.0**-127 + 2.0**-134, 3 * 2.0**-134])
    near = np.array([1 + 2**-8 + 2**-40, 1 + 2**-8 - 2**-40, 3.39e38, 3.4e38, -3.4e38])
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0**-133, 2.0**-134, 2.0**-149])
    xs = np.concatenate([rng.normal(0, 100, 20000), rng.normal(0, 1e-38, 2000),
                         rng.standard_cauchy(2000) * 1e30, ties, near, special])
    got = oracle.bf16_from_f64_np(xs)
    np.testing.assert_array_equal(got, oracle.bf16_from_f64(xs))
    finite = np.isfinite(xs)
    want = np.array([_nearest_bf16(float(v)) for v in xs[finite]])
    np.testing.assert_array_equal(oracle.bf16_to_f64(got[finite]), want)
    assert got[np.isnan(xs)][0] == 0x7FC0
    assert oracle.bf16_from_f64_np(np.array([-0.0]))[0] == 0x8000


def test_batched_dequant_matches_scalar_decode_and_nan_scale():
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, (40, 64), dtype=np.uint8)
    s = rng.integers(0, 255, (40, 4), dtype=np.uint8)
    s[3, 1] = 255
    a, b = oracle.dequant(q, s, 40, 128), oracle.dequant_np(q, s)
    np.testing.assert_array_equal(a, b)
    assert np.all(np.isnan(b[3, 32:64])) and np.all(np.isfinite(b[3, :32]))


def _tiny(bias=False, shared=False, actq=0, seed=0):
    d = synth.TINY
    wr, wi, wo = synth.host_dense(d, seed)
    ex = {e: synth.host_expert(d, seed, e) for e in range(d.n_experts)}
    b = synth.host_f32_normal(seed, synth.S_BIAS, 0, d.n_experts, 1.0) if bias else None
    sh = (*synth.host_shared(d, 2, 64, seed), 2) if shared else None
    return oracle.Layer(d, wr, wi, wo, ex, bias=b, actq=actq, shared=sh)


@pytest.mark.parametrize("actq", [0, 1, 2])
@pytest.mark.parametrize("bias,shared", [(False, False), (True, False), (True, True)])
def test_batched_forward_equals_scalar_forward_tiny(actq, bias, shared):
    lay = _tiny(bias, shared, actq)
    x = synth.host_bf16_normal(9, synth.S_X, 0, 200 * lay.d.hidden, 1.0).reshape(200, lay.d.hidden)
    a, b = lay.forward(x, nthreads=4), lay.forward_np(x, nthreads=4)
    for k in ("idx", "z", "c", "y"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_allclose(a["w"], b["w"], rtol=0, atol=0)


def test_completion_with_a_given_selection():
    """With its own selection the completion is the forward pass; with another selection it is
    the scalar steps (weights at those experts, expert rows, combine, latent out) in order."""
    lay = _tiny(bias=True)
    d = lay.d
    x = synth.host_bf16_normal(10, synth.S_X, 0, 6 * d.hidden, 1.0).reshape(6, d.hidden)
    ref = lay.forward(x)
    same = lay.forward_with_selection(x, ref["idx"])
    np.testing.assert_array_equal(same["y"], ref["y"])
    sel = ref["idx"].copy()
    for t in range(6):  # swap each token's last expert for the best unselected one
        rest = [e for e in np.argsort(-ref["logits"][t]) if e not in sel[t]]
        sel[t, -1] = rest[0]
        sel[t] = np.sort(sel[t])
    got = lay.forward_with_selection(x, sel)
    lg = oracle.router_logits(d, x, lay.wr, lay.bias)
    w = oracle.route_weights(lg, sel)
    _, z = oracle.dense_proj(lay.wi, x)
    for t in range(6):
        rows = [lay.expert_row(int(e), z[t])[0] for e in sel[t]]
        c = oracle.combine(np.stack(rows), np.arange(d.top_k, dtype=np.int32), w[t:t + 1], 1, d.top_k)
        _, y = oracle.dense_proj(lay.wo, c)
        np.testing.assert_array_equal(got["y"][t], y[0])
        assert not np.array_equal(got["y"][t], ref["y"][t])


def test_batched_forward_equals_scalar_forward_k3_tokens():
    d = synth.K3
    w = synth.WORKLOADS["prefill_4k"]
    x = synth.host_x(w, 0, 2)
    b = synth.router_bias(w)
    wr, wi, wo = synth.host_dense(d, 0)
    idx = oracle.select_topk(oracle.router_logits_np(x, wr, b), d.top_k)
    ex = {int(e): synth.host_expert(d, 0, int(e)) for e in np.unique(idx)}
    lay = oracle.Layer(d, wr, wi, wo, ex, bias=b)
    a, bb = lay.forward(x, nthreads=2), lay.forward_np(x, nthreads=4)
    for k in ("idx", "z", "c", "y"):
        np.testing.assert_array_equal(a[k], bb[k], err_msg=k)
