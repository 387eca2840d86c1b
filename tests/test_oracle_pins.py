"""Pins of the CPU oracle against facts that do not come from the oracle itself:
the format tables of the OCP MX v1.0 spec, the sizes the pages print, hand-worked cases,
library routines (numpy / scipy / torch CPU) on special cases, brute force on tiny inputs,
and exact invariants. Runs without a GPU."""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def _pow2(tok):
    if tok == "nan":
        return float("nan")
    if tok.startswith("2^"):
        return math.ldexp(1.0, int(tok[2:]))
    if "*2^" in tok:
        a, b = tok.split("*2^")
        return float(a) * math.ldexp(1.0, int(b))
    return float(tok)


# ------------------------------------------------------------------ formats
def test_e2m1_table_matches_ocp():
    for ln in _rows("e2m1_ocp_mx_v1.txt"):
        c, v = ln.split()
        got = oracle.e2m1(int(c))
        assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v)), (c, got, v)


def test_e8m0_all_256():
    gold = {int(a): _pow2(b) for a, b in (ln.split() for ln in _rows("e8m0_ocp_mx_v1.txt"))}
    for e in range(256):
        got = oracle.e8m0(e)
        want = gold.get(e, math.ldexp(1.0, e - 127) if e < 255 else float("nan"))
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, e


def test_e4m3_points_and_all_codes_vs_torch():
    for ln in _rows("e4m3_ocp_mx_v1.txt"):
        c, v = ln.split()
        got, want = oracle.e4m3(int(c, 16)), _pow2(v)
        assert (math.isnan(got) and math.isnan(want)) or got == want, (c, got, want)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_rne_vs_torch_and_saturation():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.normal(0, 30, 4000), rng.normal(0, 0.01, 2000),
                           np.array([0.0, -0.0, 448.0, -448.0, 2.0**-10, 3 * 2.0**-11])])
    vals = vals[np.abs(vals) <= 448].astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        assert oracle.e4m3_encode(float(v)) == int(r), v
    assert oracle.e4m3(oracle.e4m3_encode(500.0)) == 448.0
    assert oracle.e4m3(oracle.e4m3_encode(-1e9)) == -448.0
    assert oracle.e4m3(oracle.e4m3_encode(460.0)) == 448.0


def test_mxfp8_blocks_hand_worked():
    def expand(s):
        out = []
        for g in s.split():
            v, n = g.split("*")
            out += [float(v)] * int(n)
        return np.array(out)

    for ln in _rows("mxfp8_blocks.txt"):
        a, sc, b = [p.strip() for p in ln.split("|")]
        v = expand(a)
        codes, scale = oracle.mxfp8_block(v)
        assert scale == int(sc), ln
        want = v if b == "same" else expand(b)
        np.testing.assert_array_equal(oracle.mxfp8_roundtrip(v), want, err_msg=ln)


def _nearest_bf16_py(x):
    """Independent statement of round-to-nearest-even to 8 significant bits (normal range)."""
    if x == 0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)
    return round(m * 256) * math.ldexp(1.0, e - 8)  # Python round(): ties to even


def test_bf16_rounding():
    f = lambda x: float(oracle.bf16_to_f64(oracle.bf16_from_f64(np.array([x])))[0])
    assert f(1 + 2**-8) == 1.0                      # tie -> even
    assert f(1 + 3 * 2**-8) == 1 + 2**-6            # tie -> even (upwards)
    assert f(1 + 2**-8 + 2**-30) == 1 + 2**-7       # just above the tie: no double rounding
    assert f(-(1 + 2**-8 + 2**-30)) == -(1 + 2**-7)
    assert f(3.4e38) == math.inf and f(3.39e38) == (2 - 2**-7) * 2.0**127
    rng = np.random.default_rng(1)
    xs = rng.normal(0, 100, 3000)
    got = oracle.bf16_to_f64(oracle.bf16_from_f64(xs))
    np.testing.assert_array_equal(got, [_nearest_bf16_py(x) for x in xs])
    # float32-exact inputs: torch's float32 -> bf16 cast is RNE
    xs32 = xs.astype(np.float32)
    ref = torch.from_numpy(xs32).to(torch.bfloat16).view(torch.uint16).numpy()
    np.testing.assert_array_equal(oracle.bf16_from_f64(xs32.astype(np.float64)), ref)


TABLE = np.array([float(ln.split()[1]) for ln in _rows("e2m1_ocp_mx_v1.txt")])


def numpy_dequant(q, s):
    """Independent numpy decode: low nibble = even weight, high nibble = odd weight,
    scale byte j//32 along K."""
    q = np.asarray(q, np.uint8)
    N, KB = q.shape
    codes = np.empty((N, 2 * KB), np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    sc = np.repeat(np.ldexp(1.0, np.asarray(s, np.int64) - 127), 32, axis=1)
    return TABLE[codes] * sc


def test_nibble_order_closed_case():
    # byte 0x21: low nibble 1 -> weight 0 = 0.5, high nibble 2 -> weight 1 = 1.0
    q = np.array([0x21] + [0] * 15, np.uint8)
    s = np.array([127], np.uint8)
    assert oracle.mx_weight(q, s, 0) == 0.5
    assert oracle.mx_weight(q, s, 1) == 1.0


def test_dequant_vs_numpy_and_scale_axis():
    rng = np.random.default_rng(2)
    N, K = 6, 128
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    s = rng.integers(100, 140, (N, K // 32), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.dequant(q, s, N, K), numpy_dequant(q, s))
    for n in range(N):
        np.testing.assert_array_equal(oracle.dequant_row(q[n], s[n], K), numpy_dequant(q, s)[n])
    # scale j//32 applies to weights 32j..32j+31 only
    q1 = np.full((1, K // 2), 0x22, np.uint8)  # every weight = 1.0 * scale
    s1 = np.array([[127, 128, 129, 130]], np.uint8)
    w = oracle.dequant(q1, s1, 1, K)[0]
    np.testing.assert_array_equal(w, np.repeat([1.0, 2.0, 4.0, 8.0], 32))


def test_expert_size_arithmetic_matches_pages():
    g = {ln.split()[0]: float(ln.split()[1]) for ln in _rows("k3_sizes.txt")}
    d = synth.K3
    assert (d.n_experts, d.top_k, d.hidden, d.latent) == (g["n_experts"], g["top_k"], g["hidden"], g["latent"])
    assert oracle.expert_params(d) == g["expert_params"]
    assert oracle.expert_bytes(d) == g["expert_bytes"] == d.expert_bytes
    assert oracle.expert_bytes(d) / oracle.expert_params(d) == g["bytes_per_weight"]
    assert 8 * g["bytes_per_weight"] == g["mxfp4_bpw"]
    # the intermediate width follows from the parameter count: 33,030,144 / (3 * 3584)
    assert g["expert_params"] / (3 * g["latent"]) == d.inter == 3072
    # 82,432 x 17,547,264 B = 1.44645e12 B; the page prints 1.447 TB (within one unit of
    # its last printed digit)
    assert abs(g["routed_experts"] * oracle.expert_bytes(d) / 1e12 - g["routed_bytes_tb"]) < 1e-3
    assert abs(g["routed_experts"] * oracle.expert_params(d) / 1e9 - g["routed_params_b"]) < 0.05


# ------------------------------------------------------------------ routing
def test_topk_hand_worked():
    for ln in _rows("topk_cases.txt"):
        k, lg, want = [p.strip() for p in ln.split("|")]
        l = np.array([float(v) for v in lg.split()])[None, :]
        got = oracle.select_topk(l, int(k))[0]
        assert list(got) == [int(v) for v in want.split()], ln


def test_topk_vs_lexsort_brute_force_with_ties():
    rng = np.random.default_rng(3)
    T, E, k = 40, 64, 8
    lg = rng.integers(-5, 6, (T, E)).astype(np.float64)  # many exact ties
    got = oracle.select_topk(lg, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t]))  # primary -l, secondary index
        assert list(got[t]) == sorted(order[:k].tolist())


def test_route_weights_special_cases():
    rng = np.random.default_rng(4)
    T, E = 5, 16
    lg = rng.normal(0, 2, (T, E))
    full = oracle.select_topk(lg, E)
    np.testing.assert_allclose(oracle.route_weights(lg, full), scipy.special.softmax(lg, axis=1),
                               rtol=1e-14, atol=0)
    one = oracle.select_topk(lg, 1)
    assert np.all(oracle.route_weights(lg, one) == 1.0)
    idx = oracle.select_topk(lg, 4)
    w = oracle.route_weights(lg, idx)
    want = scipy.special.softmax(np.take_along_axis(lg, idx, 1), axis=1)
    np.testing.assert_allclose(w, want, rtol=1e-13)


def test_router_logits_vs_numpy_with_bias():
    d = synth.TINY
    rng = np.random.default_rng(6)
    x = synth.host_bf16_normal(9, 1, 0, 3 * d.hidden, 1.0).reshape(3, d.hidden)
    wr = synth.host_bf16_normal(9, 2, 0, d.n_experts * d.hidden, 0.02).reshape(d.n_experts, d.hidden)
    b = rng.normal(0, 1, d.n_experts).astype(np.float32)
    got = oracle.router_logits(d, x, wr, b)
    want = oracle.bf16_to_f64(x) @ oracle.bf16_to_f64(wr).T + b.astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.router_logits_np(x, wr, b), got, rtol=1e-12, atol=1e-12)


def test_permute_vs_sorted_brute_force():
    E = 13
    for T, k, skew in [(1, 4, "uniform"), (17, 4, "uniform"), (9, 3, "one"), (30, 5, "zipf")]:
        idx = synth.host_topk_sets(7, T, E, k, skew)
        off, rt, rs, sr = oracle.permute(idx, E)
        pairs = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
        assert [p[1] for p in pairs] == rt.tolist()
        assert [p[2] for p in pairs] == rs.tolist()
        counts = np.bincount(idx.ravel(), minlength=E)
        assert off.tolist() == [0] + np.cumsum(counts).tolist()
        for r, (e, t, j) in enumerate(pairs):
            assert sr[t * k + j] == r and off[e] <= r < off[e + 1]


def test_dense_proj_vs_numpy():
    rng = np.random.default_rng(8)
    W = synth.host_bf16_normal(1, 3, 0, 48 * 96, 0.02).reshape(48, 96)
    x = synth.host_bf16_normal(1, 1, 0, 5 * 96, 1.0).reshape(5, 96)
    out, ob = oracle.dense_proj(W, x)
    want = oracle.bf16_to_f64(x) @ oracle.bf16_to_f64(W).T
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(oracle.bf16_to_f64(ob), [[_nearest_bf16_py(v) for v in r] for r in want])


# ------------------------------------------------------------------ expert FFN and layer
def tiny_layer(seed=0, experts=None, bias=None, actq=0):
    d = synth.TINY
    wr, wi, wo = synth.host_dense(d, seed)
    ex = experts if experts is not None else {e: synth.host_expert(d, seed, e) for e in range(d.n_experts)}
    return oracle.Layer(d, wr, wi, wo, ex, bias=bias, actq=actq), ex


def _silu(g):
    return g / (1.0 + np.exp(-g))


def numpy_layer(d, wr, wi, wo, ex, x, bias=None):
    """Independent numpy statement of the layer on the tiny config."""
    xf = oracle.bf16_to_f64(x)
    lg = xf @ oracle.bf16_to_f64(wr).T + (0 if bias is None else bias.astype(np.float64))
    T, E = lg.shape
    k = d.top_k
    idx = np.stack([np.sort(np.lexsort((np.arange(E), -lg[t]))[:k]) for t in range(T)])
    p = scipy.special.softmax(lg, axis=1)
    sel = np.take_along_axis(p, idx, 1)
    w = sel / sel.sum(1, keepdims=True)
    nb = np.vectorize(_nearest_bf16_py)
    z = nb(xf @ oracle.bf16_to_f64(wi).T)
    y = np.empty((T, d.hidden))
    for t in range(T):
        c = np.zeros(d.latent)
        for j in range(k):
            e = idx[t, j]
            G = numpy_dequant(ex[e]["gate_q"], ex[e]["gate_s"])
            U = numpy_dequant(ex[e]["up_q"], ex[e]["up_s"])
            D = numpy_dequant(ex[e]["down_q"], ex[e]["down_s"])
            a = nb(_silu(G @ z[t]) * (U @ z[t]))
            c += w[t, j] * (D @ a)
        y[t] = nb(oracle.bf16_to_f64(oracle.bf16_from_f64(nb(c))) @ oracle.bf16_to_f64(wo).T)
    return idx, w, z, y


@pytest.mark.parametrize("with_bias", [False, True])
def test_tiny_layer_vs_numpy(with_bias):
    d = synth.TINY
    bias = np.random.default_rng(11).normal(0, 1, d.n_experts).astype(np.float32) if with_bias else None
    layer, ex = tiny_layer(bias=bias)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    r = layer.forward(x, nthreads=2)
    wr, wi, wo = synth.host_dense(d, 0)
    idx, w, z, y = numpy_layer(d, wr, wi, wo, ex, x, bias)
    np.testing.assert_array_equal(r["idx"], idx)
    np.testing.assert_allclose(r["w"], w, rtol=1e-12)
    np.testing.assert_array_equal(oracle.bf16_to_f64(r["z"]), z)
    # same roundings; only double summation order differs -> rare 1-ulp bf16 straddles
    yo = oracle.bf16_to_f64(r["y"])
    rel = np.linalg.norm(yo - y, axis=1) / np.linalg.norm(y, axis=1)
    assert rel.max() < 1e-6, rel


def test_tiny_layer_detects_transposed_down():
    """A transposed expert matrix (a layout mistake) must change the result."""
    d = synth.TINY
    layer, ex = tiny_layer()
    x = synth.host_x(synth.WORKLOADS["tiny"])
    good = oracle.bf16_to_f64(layer.forward(x)["y"])
    bad_ex = {}
    for e, t in ex.items():
        t2 = dict(t)
        D = numpy_dequant(t["down_q"], t["down_s"])
        # rebuild a down matrix whose codes are the transpose of the original codes
        codes = np.empty((d.latent, d.inter), np.uint8)
        codes[:, 0::2] = t["down_q"] & 0xF
        codes[:, 1::2] = t["down_q"] >> 4
        ct = codes.T.copy().reshape(d.latent, d.inter) if d.latent == d.inter else None
        if ct is None:
            pytest.skip("non-square")
        t2["down_q"] = (ct[:, 0::2] | (ct[:, 1::2] << 4)).astype(np.uint8)
        bad_ex[e] = t2
    bad_layer, _ = tiny_layer(experts=bad_ex)
    bad = oracle.bf16_to_f64(bad_layer.forward(x)["y"])
    cos = np.sum(good * bad) / (np.linalg.norm(good) * np.linalg.norm(bad))
    assert cos < 0.5


def test_invariant_zero_codes_give_zero():
    d = synth.TINY
    ex = {e: {n: (np.zeros_like(a) if n.endswith("_q") else a) for n, a in synth.host_expert(d, 0, e).items()}
          for e in range(d.n_experts)}
    layer, _ = tiny_layer(experts=ex)
    y = layer.forward(synth.host_x(synth.WORKLOADS["tiny"]))["y"]
    assert np.all(oracle.bf16_to_f64(y) == 0.0)


def test_invariant_up_scale_plus_one_doubles_output_exactly():
    d = synth.TINY
    base = {e: synth.host_expert(d, 0, e) for e in range(d.n_experts)}
    dbl = {e: dict(t, up_s=(t["up_s"] + 1).astype(np.uint8)) for e, t in base.items()}
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y1 = oracle.bf16_to_f64(tiny_layer(experts=base)[0].forward(x)["y"])
    y2 = oracle.bf16_to_f64(tiny_layer(experts=dbl)[0].forward(x)["y"])
    np.testing.assert_array_equal(y2, 2 * y1)


def test_invariant_one_hot_code_closed_form():
    d = synth.TINY
    L, I = d.latent, d.inter
    e, n, kk, m = 3, 5, 7, 9  # gate/up row n, input position kk; down column n -> row m
    t = {
        "gate_q": np.zeros((I, L // 2), np.uint8), "gate_s": np.full((I, L // 32), 127, np.uint8),
        "up_q": np.zeros((I, L // 2), np.uint8), "up_s": np.full((I, L // 32), 128, np.uint8),
        "down_q": np.zeros((L, I // 2), np.uint8), "down_s": np.full((L, I // 32), 126, np.uint8),
    }
    t["gate_q"][n, kk // 2] = 0x5 << (4 * (kk % 2))    # gate weight 3.0 * 2^0
    t["up_q"][n, kk // 2] = 0x4 << (4 * (kk % 2))      # up weight 2.0 * 2^1 = 4
    t["down_q"][m, n // 2] = 0xB << (4 * (n % 2))      # down weight -1.5 * 2^-1 = -0.75
    layer, _ = tiny_layer(experts={e: t})
    z = synth.host_bf16_normal(4, 1, 0, L, 1.0)
    o, a = layer.expert_row(e, z)
    zk = float(oracle.bf16_to_f64(z[kk:kk + 1])[0])
    g, u = 3.0 * zk, 4.0 * zk
    a_n = _nearest_bf16_py(g / (1 + math.exp(-g)) * u)
    want = np.zeros(L)
    want[m] = -0.75 * a_n
    np.testing.assert_array_equal(o, want)


def test_invariant_token_permutation():
    layer, _ = tiny_layer()
    x = synth.host_x(synth.WORKLOADS["tiny"])
    perm = np.array([5, 2, 7, 0, 1, 6, 3, 4])
    a, b = layer.forward(x), layer.forward(x[perm])
    np.testing.assert_array_equal(b["y"], a["y"][perm])
    np.testing.assert_array_equal(b["idx"], a["idx"][perm])


def test_mxfp8_mode_expert_row_vs_numpy():
    d = synth.TINY
    layer, ex = tiny_layer(actq=1)
    z = synth.host_bf16_normal(3, 1, 0, d.latent, 1.0)
    e = 2
    o, a = layer.expert_row(e, z)
    zq = oracle.mxfp8_roundtrip(oracle.bf16_to_f64(z))
    G, U, D = (numpy_dequant(ex[e][p + "_q"], ex[e][p + "_s"]) for p in ("gate", "up", "down"))
    a_ref = np.vectorize(_nearest_bf16_py)(_silu(G @ zq) * (U @ zq))
    np.testing.assert_array_equal(oracle.bf16_to_f64(a), a_ref)
    np.testing.assert_allclose(o, D @ oracle.mxfp8_roundtrip(a_ref), rtol=1e-12, atol=1e-9)


def test_combine_vs_numpy():
    rng = np.random.default_rng(12)
    T, k, L = 4, 3, 64
    o = rng.normal(0, 100, (T * k, L))
    sr = rng.permutation(T * k).astype(np.int32)
    w = rng.dirichlet(np.ones(k), T)
    c = oracle.combine(o, sr, w, T, k)
    for t in range(T):
        ref = sum(w[t, j] * o[sr[t * k + j]] for j in range(k))
        np.testing.assert_array_equal(oracle.bf16_to_f64(c[t]), [_nearest_bf16_py(v) for v in ref])
