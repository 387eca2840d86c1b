"""GPU parity of the routing half of the layer: the device input generator, router logits +
top-k (k3moe_route) and the token-by-expert permutation (k3moe_permute), against the oracle.

Indices and permutations are compared bit for bit. Where fp32 router logits decide a
selection (random-normal inputs), tokens whose oracle logits tie within the fp32 error at
the top-k boundary are checked for validity instead; a separate integer-exact router case
gives identical logits on both sides and must match exactly, ties included."""
import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth
from k3help import (DEV, LOGIT_ATOL, LOGIT_RTOL, dims, up, stream, workspace, check_ok,
                    topk_gap_ambiguous, selection_valid)

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host():
    d = synth.TINY
    n = d.n_experts * d.gate_q_bytes
    t = torch.empty(n, dtype=torch.uint8, device=DEV)
    synth.dev_bytes(0, synth.S_GATE_Q, 0, n, t.data_ptr(), stream())
    np.testing.assert_array_equal(t.cpu().numpy(), synth.host_bytes(0, synth.S_GATE_Q, 0, n))
    # ragged offset / length (unaligned path)
    t2 = torch.empty(1001, dtype=torch.uint8, device=DEV)
    synth.dev_bytes(3, 9, 13, 1001, t2.data_ptr(), stream())
    np.testing.assert_array_equal(t2.cpu().numpy(), synth.host_bytes(3, 9, 13, 1001))
    t3 = torch.empty(5000, dtype=torch.uint8, device=DEV)
    synth.dev_uniform_u8(0, synth.S_UP_S, 777, 5000, 120, 127, t3.data_ptr(), stream())
    np.testing.assert_array_equal(t3.cpu().numpy(), synth.host_uniform_u8(0, synth.S_UP_S, 777, 5000, 120, 127))
    t4 = torch.empty(7000, dtype=torch.int16, device=DEV)
    synth.dev_bf16_normal(2, synth.S_W_IN, 12345, 7000, 0.02, t4.data_ptr(), stream())
    np.testing.assert_array_equal(t4.cpu().numpy().view(np.uint16),
                                  synth.host_bf16_normal(2, synth.S_W_IN, 12345, 7000, 0.02))


def _route(d, x_np, wr_np, bias=None, T=None, logits_out=True):
    dm = dims(d)
    T = x_np.shape[0] if T is None else T
    x, wr = up(x_np), up(wr_np)
    b = None if bias is None else up(np.asarray(bias, np.float32))
    lg = torch.empty((max(T, 1), d.n_experts), dtype=torch.float32, device=DEV)
    idx = torch.empty((max(T, 1), d.top_k), dtype=torch.int32, device=DEV)
    w = torch.empty((max(T, 1), d.top_k), dtype=torch.float32, device=DEV)
    ws, n = workspace(dm, T)
    k3.k3moe_route(dm, x.data_ptr(), T, wr.data_ptr(), None if b is None else b.data_ptr(),
                   lg.data_ptr() if logits_out else None, idx.data_ptr(), w.data_ptr(), ws.data_ptr(), n,
                   stream())
    check_ok(ws)
    return lg.cpu().numpy()[:T], idx.cpu().numpy()[:T], w.cpu().numpy()[:T]


@pytest.mark.parametrize("name,T,bias", [("tiny", 8, None), ("k3", 1, None), ("k3", 64, "normal"),
                                         ("k3", 300, "zipf"), ("k3", 2048, "zipf")])
def test_route_random_normal(name, T, bias):
    d = synth.TINY if name == "tiny" else synth.K3
    x = synth.host_bf16_normal(5, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    wr = synth.host_bf16_normal(5, synth.S_W_ROUTER, 0, d.n_experts * d.hidden, 0.02).reshape(d.n_experts, d.hidden)
    b = None
    if bias == "normal":
        b = synth.host_f32_normal(5, synth.S_BIAS, 0, d.n_experts, 1.0)
    elif bias == "zipf":
        b = synth.zipf_bias(d.n_experts, 5)
    lg, idx, w = _route(d, x, wr, b)
    ref_lg = oracle.router_logits_np(x, wr, b)
    tol = LOGIT_ATOL + LOGIT_RTOL * np.abs(ref_lg)
    assert np.all(np.abs(lg - ref_lg) <= tol), np.abs(lg - ref_lg).max()
    ref_idx = oracle.select_topk(ref_lg, d.top_k)
    amb = topk_gap_ambiguous(ref_lg, d.top_k, 2 * (LOGIT_ATOL + LOGIT_RTOL * np.abs(ref_lg).max()))
    same = np.all(idx == ref_idx, axis=1)
    assert np.all(same | amb), f"{(~same & ~amb).sum()} unambiguous tokens differ"
    for t in np.nonzero(~same)[0]:
        assert selection_valid(ref_lg[t], idx[t], d.top_k, 4 * LOGIT_ATOL + 4 * LOGIT_RTOL * np.abs(ref_lg[t]).max())
    assert np.all(np.diff(idx, axis=1) > 0)  # ascending
    ref_w = oracle.route_weights(ref_lg, ref_idx)
    np.testing.assert_allclose(w[same], ref_w[same], rtol=5e-4, atol=1e-6)


def test_route_integer_exact_with_ties():
    """Small-integer router and tokens: every product and partial sum is exact in fp32, so
    both sides see identical logits; duplicated router rows create exact ties, which must
    resolve to the lowest index."""
    d = synth.Dims(hidden=256, latent=128, inter=128, n_experts=96, top_k=8)
    rng = np.random.default_rng(0)
    xs = rng.integers(-2, 3, (40, d.hidden)).astype(np.float32)
    ws_ = (rng.integers(-3, 4, (d.n_experts, d.hidden)) * 0.0625).astype(np.float32)
    ws_[10] = ws_[3]
    ws_[50] = ws_[3]
    ws_[77] = ws_[20]
    xs[5] = 0  # all logits equal (zero) -> experts 0..k-1
    to_bf16 = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    x, wr = to_bf16(xs), to_bf16(ws_)
    lg, idx, w = _route(d, x, wr)
    ref_lg = oracle.router_logits(d, x, wr)
    np.testing.assert_array_equal(lg.astype(np.float64), ref_lg)
    np.testing.assert_array_equal(idx, oracle.select_topk(ref_lg, d.top_k))
    assert list(idx[5]) == list(range(d.top_k))
    np.testing.assert_allclose(w, oracle.route_weights(ref_lg, oracle.select_topk(ref_lg, d.top_k)),
                               rtol=2e-6, atol=1e-7)


def test_route_ties_across_expert_groups_and_nan():
    """The selection's order on exact logits (the routing rule: the k largest logits, equal
    logits to the lower expert index, NaN below every number) on 896 experts, with tie groups
    that straddle the device's 128-expert sort groups. Integer router weights and one-hot
    tokens make every logit exact on both sides."""
    d = synth.Dims(hidden=128, latent=64, inter=64, n_experts=896, top_k=16)
    E, H = d.n_experts, d.hidden
    wr = np.zeros((E, H), np.float32)
    wr[:, 0] = 1.0
    wr[100:140, 0] = 2.0                 # token 1: a 40-way tie across the group at 128
    wr[125:132, 1] = 3.0                 # token 2: 7 above the rest, across 128 ...
    wr[0:E:50, 1] = 2.0                  # ... then the lowest 9 of an 18-way tie
    wr[5, :] = -1.0                      # token 0 (x = 0): every finite logit 0
    wr[3, :] = np.nan                    # every token: expert 3's logit is NaN
    xs = np.zeros((4, H), np.float32)
    xs[1, 0] = 1.0
    xs[2, 1] = 1.0
    xs[3, 2] = np.nan                    # token 3: every logit NaN -> the lowest k indices
    to_bf16 = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    lg, idx, w = _route(d, to_bf16(xs), to_bf16(wr))
    want = [
        [0, 1, 2] + list(range(4, 17)),
        list(range(100, 116)),
        sorted(list(range(125, 132)) + list(range(0, 450, 50))),
        list(range(16)),
    ]
    for t in range(4):
        assert list(idx[t]) == want[t], (t, list(idx[t]))
    ref_lg = oracle.router_logits(d, to_bf16(xs), to_bf16(wr))
    np.testing.assert_array_equal(idx, oracle.select_topk(ref_lg, d.top_k))
    # weights: softmax over the kept logits (equal to softmax over all renormalised, for finite logits)
    for t in range(3):
        kept = ref_lg[t, idx[t]]
        e = np.exp(kept - kept.max())
        np.testing.assert_allclose(w[t], e / e.sum(), rtol=2e-6)


@pytest.mark.parametrize("k", [1, 32])
def test_route_k_edge(k):
    d = synth.Dims(hidden=128, latent=64, inter=64, n_experts=32, top_k=k)
    x = synth.host_bf16_normal(1, 1, 0, 5 * d.hidden, 1.0).reshape(5, d.hidden)
    wr = synth.host_bf16_normal(1, 2, 0, d.n_experts * d.hidden, 0.5).reshape(d.n_experts, d.hidden)
    lg, idx, w = _route(d, x, wr)
    ref_lg = oracle.router_logits(d, x, wr)
    if k == 1:
        assert np.all(w == 1.0)
        np.testing.assert_array_equal(idx, oracle.select_topk(ref_lg, 1))
    else:  # k = E: every expert, weights = full softmax
        np.testing.assert_array_equal(idx, np.tile(np.arange(32), (5, 1)))
        np.testing.assert_allclose(w, oracle.route_weights(ref_lg, oracle.select_topk(ref_lg, 32)),
                                   rtol=1e-5)


def test_route_zero_tokens():
    d = synth.TINY
    _route(d, np.zeros((1, d.hidden), np.uint16), np.zeros((d.n_experts, d.hidden), np.uint16), T=0)


def _permute(d, idx_np):
    dm = dims(d)
    T = idx_np.shape[0]
    idx = up(idx_np.astype(np.int32)) if T else torch.zeros((1, d.top_k), dtype=torch.int32, device=DEV)
    rows = max(T * d.top_k, 1)
    off = torch.empty(d.n_experts + 1, dtype=torch.int32, device=DEV)
    rt, rs, sr = (torch.empty(rows, dtype=torch.int32, device=DEV) for _ in range(3))
    ws, n = workspace(dm, T)
    k3.k3moe_permute(dm, idx.data_ptr(), T, off.data_ptr(), rt.data_ptr(), rs.data_ptr(),
                     sr.data_ptr(), ws.data_ptr(), n, stream())
    check_ok(ws)
    return off.cpu().numpy(), rt.cpu().numpy()[:T * d.top_k], rs.cpu().numpy()[:T * d.top_k], \
        sr.cpu().numpy()[:T * d.top_k]


@pytest.mark.parametrize("T,skew", [(1, "uniform"), (7, "uniform"), (64, "one"), (256, "zipf"),
                                    (257, "uniform"), (1000, "zipf"), (4096, "zipf")])
def test_permute_bit_exact(T, skew):
    d = synth.K3
    idx = synth.host_topk_sets(T, T, d.n_experts, d.top_k, skew)
    got = _permute(d, idx)
    want = oracle.permute(idx, d.n_experts)
    for g, w_ in zip(got, want):
        np.testing.assert_array_equal(g, w_)


def test_permute_large_and_tiny():
    d = synth.K3
    T = 32768
    rng = np.random.default_rng(9)
    # fast synthetic sets for a large T: distinct experts per token via random permutations
    idx = np.sort(np.argsort(rng.random((T, d.n_experts)), axis=1)[:, :d.top_k], axis=1).astype(np.int32)
    got = _permute(d, idx)
    want = oracle.permute(idx, d.n_experts)
    for g, w_ in zip(got, want):
        np.testing.assert_array_equal(g, w_)
    dt = synth.TINY
    idx = synth.host_topk_sets(2, 8, dt.n_experts, dt.top_k, "uniform")
    for g, w_ in zip(_permute(dt, idx), oracle.permute(idx, dt.n_experts)):
        np.testing.assert_array_equal(g, w_)


def test_permute_deterministic_reruns():
    d = synth.K3
    idx = synth.host_topk_sets(11, 600, d.n_experts, d.top_k, "zipf")
    first = _permute(d, idx)
    for _ in range(5):
        for a, b in zip(first, _permute(d, idx)):
            np.testing.assert_array_equal(a, b)
