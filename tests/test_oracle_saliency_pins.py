"""Pins of the oracle's REAP saliency ("kimi-k3-mlx" digest, REAP pruning section:
S_j = (1/|C|) sum_x g_j(x) * ||e_j(x)||_2) against what the formula fixes by itself. Runs
without a GPU."""
import numpy as np

import oracle
import synth


def _tiny(k=4, up_shift=0, zero=False, bias=None, seed=0):
    d = synth.Dims(hidden=256, latent=128, inter=128, n_experts=32, top_k=k)
    wr, wi, wo = synth.host_dense(d, seed)
    ex = {}
    for e in range(d.n_experts):
        t = synth.host_expert(d, seed, e)
        if up_shift:
            t["up_s"] = (t["up_s"] + up_shift).astype(np.uint8)
        if zero:
            t = {n: (np.zeros_like(a) if n.endswith("_q") else a) for n, a in t.items()}
        ex[e] = t
    return oracle.Layer(d, wr, wi, wo, ex, bias=bias)


X = synth.host_bf16_normal(7, synth.S_X, 0, 40 * 256, 1.0).reshape(40, 256)


def test_saliency_matches_its_definition_by_brute_force():
    lay = _tiny()
    d = lay.d
    S = oracle.saliency(lay, X, nthreads=2)
    ref = lay.forward(X)  # the scalar statement: its selection and weights
    want = np.zeros(d.n_experts)
    _, z = oracle.dense_proj(lay.wi, X)
    for t in range(X.shape[0]):
        for j in range(d.top_k):
            e = int(ref["idx"][t, j])
            o, _ = lay.expert_row(e, z[t])
            want[e] += ref["w"][t, j] * np.sqrt(np.sum(o * o))
    want /= X.shape[0]
    np.testing.assert_allclose(S, want, rtol=1e-12, atol=0)
    assert np.all(S[np.setdiff1d(np.arange(d.n_experts), ref["idx"])] == 0)  # never selected -> 0


def test_saliency_zero_experts_give_zero():
    assert np.all(oracle.saliency(_tiny(zero=True), X) == 0)


def test_saliency_doubles_exactly_with_the_up_scales():
    """+1 on every up exponent doubles every GLU output and so every expert output: S doubles
    exactly (the selection and the weights do not depend on the experts)."""
    a = oracle.saliency(_tiny(), X)
    b = oracle.saliency(_tiny(up_shift=1), X)
    np.testing.assert_array_equal(b, 2 * a)


def test_saliency_with_one_expert_per_token_is_the_mean_output_norm():
    """k = 1: g_j(x) = 1 for the one selected expert, so S_j is the sum of that expert's
    output norms over its tokens, divided by |C|."""
    lay = _tiny(k=1)
    S = oracle.saliency(lay, X)
    ref = lay.forward_np(X)
    norms = np.linalg.norm(ref["o"][:, 0], axis=1)
    for e in range(lay.d.n_experts):
        np.testing.assert_allclose(S[e], norms[ref["idx"][:, 0] == e].sum() / X.shape[0], rtol=1e-13)


def test_saliency_is_a_mean_over_the_calibration_tokens():
    """Token order does not matter, and the set C twice gives the same mean."""
    lay = _tiny()
    a = oracle.saliency(lay, X)
    perm = np.random.default_rng(0).permutation(X.shape[0])
    np.testing.assert_allclose(oracle.saliency(lay, X[perm]), a, rtol=1e-13)
    np.testing.assert_allclose(oracle.saliency(lay, np.concatenate([X, X])), a, rtol=1e-13)


def test_saliency_weights_sum_to_one_per_token():
    """With every expert's output norm forced equal (checked through the accumulator itself),
    sum_j S_j = that norm: the renormalised weights of a token sum to one."""
    d = _tiny().d
    T = 10
    idx = np.tile(np.arange(d.top_k, dtype=np.int32), (T, 1))
    w = np.random.default_rng(1).dirichlet(np.ones(d.top_k), T)
    o = np.zeros((T, d.top_k, d.latent))
    o[:, :, 0] = 3.0  # ||o|| = 3 for every row
    S = oracle.saliency_accumulate(d, idx, w, o) / T
    np.testing.assert_allclose(S.sum(), 3.0, rtol=1e-14)
