"""GPU parity of the expert half and of the whole layer against the oracle: dense projection
(k3moe_project), routed expert FFN (k3moe_expert_ffn_mxfp4), combine (k3moe_combine) and
k3moe_layer_forward, on the tiny layer (every token) and on K3-sized layers (sampled tokens,
each recomputed independently by the oracle)."""
import os
import time

import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth
from k3help import (DEV, REL_L2, DeviceLayer, bf16_np, dims, up, stream, workspace, check_ok, rel_l2_rows,
                    compare_layer, run_layer)

pytestmark = pytest.mark.gpu
NCPU = os.cpu_count() or 4


@pytest.fixture(scope="module")
def k3_layer():
    lay = DeviceLayer(synth.K3, seed=0)
    torch.cuda.synchronize()
    yield lay
    del lay
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ projection
@pytest.mark.parametrize("T,N,K", [(1, 3584, 7168), (5, 128, 256), (64, 7168, 3584), (200, 192, 320),
                                   (2500, 1024, 1088), (2300, 1152, 320)])
def test_project(T, N, K):
    W = synth.host_bf16_normal(1, 3, 0, N * K, 0.02).reshape(N, K)
    x = synth.host_bf16_normal(1, 1, 0, T * K, 1.0).reshape(T, K)
    out = torch.empty((T, N), dtype=torch.int16, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    Wd, xd = up(W), up(x)  # keep the device copies alive until the kernels have run
    k3.k3moe_project(Wd.data_ptr(), xd.data_ptr(), T, N, K, out.data_ptr(), ws.data_ptr(), 256,
                     stream())
    check_ok(ws)
    got = bf16_np(out)
    want_exact, want_b = oracle.dense_proj(W, x)
    want = oracle.bf16_to_f64(want_b)
    # bf16 rounding (half an ulp, 2^-9 relative) of an fp32 sum whose error is bounded by
    # K * 2^-24 * sum |W x| (fp32 accumulation, any order)
    mag = np.abs(oracle.bf16_to_f64(x)) @ np.abs(oracle.bf16_to_f64(W)).T
    bound = np.abs(want_exact) * 2.0**-8 + K * 2.0**-24 * mag * 1.01
    assert np.all(np.abs(got - want_exact) <= bound)
    assert rel_l2_rows(got, want_exact).max() < 4e-3
    assert (got != want).mean() < 0.02


# ------------------------------------------------------------------ expert FFN
def _expert_ffn(lay, z_np, idx_np, actq=0):
    d = lay.d
    dm = dims(d, actq)
    T = z_np.shape[0]
    off, rt, rs, sr = oracle.permute(idx_np, d.n_experts)  # permutation from the host side
    o = torch.empty((T * d.top_k, d.latent), dtype=torch.float32, device=DEV)
    ws, n = workspace(dm, T)
    zd, offd, rtd = up(z_np), up(off), up(rt)
    k3.k3moe_expert_ffn_mxfp4(dm, lay.weights, zd.data_ptr(), T, offd.data_ptr(), rtd.data_ptr(),
                              o.data_ptr(), ws.data_ptr(), n, stream())
    check_ok(ws)
    return o.cpu().numpy().astype(np.float64), (off, rt, rs, sr)


# T >= 65 runs the tensor-core kernel with the weights on the MMA's M side (chunks of up to 112
# sorted rows); smaller T the one with the weights on N (chunks of up to 8), whose down pass needs
# latent % 256 == 0 (latent = 128 keeps the M-side kernel for it). DEEP has eight K stages per
# item and fewer items than SMs.
WIDE = synth.Dims(hidden=256, latent=256, inter=256, n_experts=16, top_k=4)
DEEP = synth.Dims(hidden=256, latent=1024, inter=1024, n_experts=8, top_k=2)
DIMS = {"tiny": synth.TINY, "wide": WIDE, "deep": DEEP}


@pytest.mark.parametrize("dname,T", [("tiny", 24), ("tiny", 100), ("wide", 7), ("wide", 200), ("wide", 700),
                                     ("deep", 3), ("deep", 20)])
@pytest.mark.parametrize("actq", [0, 1, 2])
def test_expert_ffn_tiny_all_rows(actq, dname, T):
    """actq 2 (MXFP4 activations, kind::mxf4) needs latent and inter multiples of 256: the tiny
    shape is refused with K3MOE_E_MODE; the wide and deep shapes run it at 8-row and many-token
    chunks. wide at 700 tokens gives experts of several hundred rows: full chunks of 112 (bf16),
    224 (MXFP8) and 192 rows (MXFP4, whose second 128-row block of activation scales only such
    chunks use)."""
    d = DIMS[dname]
    if actq == 2 and d.latent % 256:
        ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
        st = k3.k3moe_expert_ffn_mxfp4(dims(d, 2), k3.Weights(), 16, 1, 16, 16, 16, ws.data_ptr(), 256, stream(),
                                       check=False)
        assert st == 5  # K3MOE_E_MODE
        return
    lay = DeviceLayer(d, seed=0, actq=actq)
    z = synth.host_bf16_normal(3, synth.S_X, 0, T * d.latent, 1.7).reshape(T, d.latent)
    idx = synth.host_topk_sets(4, T, d.n_experts, d.top_k, "zipf")
    o, (off, rt, rs, sr) = _expert_ffn(lay, z, idx, actq)
    ol = lay.oracle(actq=actq)
    want = np.stack([ol.expert_row(int(idx[rt[r], rs[r]]), z[rt[r]])[0] for r in range(T * d.top_k)])
    err = rel_l2_rows(o, want)
    assert err.max() <= REL_L2, err.max()


@pytest.mark.parametrize("T", [5, 70])
def test_expert_ffn_gemv_path_all_rows(T):
    """inter = 192 is not a multiple of 128, so the expert GEMV runs instead of the MMA path."""
    d = synth.Dims(hidden=256, latent=128, inter=192, n_experts=32, top_k=4)
    lay = DeviceLayer(d, seed=5)
    z = synth.host_bf16_normal(6, synth.S_X, 0, T * d.latent, 1.7).reshape(T, d.latent)
    idx = synth.host_topk_sets(7, T, d.n_experts, d.top_k, "zipf")
    o, (off, rt, rs, sr) = _expert_ffn(lay, z, idx)
    ol = lay.oracle()
    want = np.stack([ol.expert_row(int(idx[rt[r], rs[r]]), z[rt[r]])[0] for r in range(T * d.top_k)])
    assert rel_l2_rows(o, want).max() <= REL_L2


@pytest.mark.parametrize("T,actq", [(40, 0), (40, 1), (40, 2), (96, 0), (96, 1), (96, 2)])
def test_expert_ffn_k3_sampled_rows(k3_layer, T, actq):
    d = synth.K3
    z = synth.host_bf16_normal(7, synth.S_X, 0, T * d.latent, 1.7).reshape(T, d.latent)
    idx = synth.host_topk_sets(8, T, d.n_experts, d.top_k, "zipf")  # skewed: multi-chunk experts
    o, (off, rt, rs, sr) = _expert_ffn(k3_layer, z, idx, actq)
    rng = np.random.default_rng(0)
    rows = sorted(set(rng.choice(T * d.top_k, 12, replace=False).tolist()) | {0, T * d.top_k - 1})
    ol = k3_layer.oracle(experts={int(idx[rt[r], rs[r]]) for r in rows}, actq=actq)
    for r in rows:
        want = ol.expert_row(int(idx[rt[r], rs[r]]), z[rt[r]])[0]
        assert rel_l2_rows(o[r], want) <= REL_L2, (r, rel_l2_rows(o[r], want))


@pytest.mark.parametrize("dname,T,actq", [("tiny", 8, 0), ("tiny", 80, 0), ("wide", 80, 0), ("deep", 5, 0),
                                          ("wide", 6, 2), ("wide", 80, 2), ("deep", 5, 2)])
def test_expert_ffn_invariants_bit_exact(dname, T, actq):
    """All-zero codes give exactly 0; +1 on every up exponent doubles every output exactly (in
    MXFP4 mode too: the GLU output doubles, its block exponents rise by one, its codes stay)."""
    d = DIMS[dname]
    z = synth.host_bf16_normal(2, synth.S_X, 0, T * d.latent, 1.0).reshape(T, d.latent)
    idx = synth.host_topk_sets(5, T, d.n_experts, d.top_k, "uniform")
    base = {e: synth.host_expert(d, 0, e) for e in range(d.n_experts)}
    zero = {e: {n: (np.zeros_like(a) if n.endswith("_q") else a) for n, a in t.items()} for e, t in base.items()}
    dbl = {e: dict(t, up_s=(t["up_s"] + 1).astype(np.uint8)) for e, t in base.items()}
    o0, _ = _expert_ffn(DeviceLayer(d, experts=zero, actq=actq), z, idx, actq)
    assert np.all(o0 == 0.0)
    o1, _ = _expert_ffn(DeviceLayer(d, experts=base, actq=actq), z, idx, actq)
    o2, _ = _expert_ffn(DeviceLayer(d, experts=dbl, actq=actq), z, idx, actq)
    np.testing.assert_array_equal(o2, 2 * o1)


@pytest.mark.parametrize("dname,T", [("tiny", 4), ("tiny", 72), ("wide", 72), ("deep", 4)])
def test_expert_ffn_nan_scale_gives_nonfinite(dname, T):
    d = DIMS[dname]
    base = {e: synth.host_expert(d, 0, e) for e in range(d.n_experts)}
    base[0]["down_s"] = base[0]["down_s"].copy()
    base[0]["down_s"][:, 0] = 255
    idx = np.tile(np.arange(d.top_k, dtype=np.int32), (T, 1))
    z = synth.host_bf16_normal(2, synth.S_X, 0, T * d.latent, 1.0).reshape(T, d.latent)
    o, (off, rt, rs, sr) = _expert_ffn(DeviceLayer(d, experts=base), z, idx)
    rows0 = np.arange(off[0], off[1])
    assert np.all(~np.isfinite(o[rows0]).all(axis=1))
    assert np.all(np.isfinite(o[off[1]:]))


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("k", [16, 1, 24, 32])  # k <= 16 and k > 16 take different kernel instances
def test_combine(k):
    import dataclasses
    d = dataclasses.replace(synth.K3, top_k=k)
    T = 33
    rng = np.random.default_rng(1)
    o = rng.normal(0, 1e5, (T * d.top_k, d.latent)).astype(np.float32)
    sr = rng.permutation(T * d.top_k).astype(np.int32)
    w = rng.dirichlet(np.ones(d.top_k), T).astype(np.float32)
    c = torch.empty((T, d.latent), dtype=torch.int16, device=DEV)
    od, srd, wd = up(o), up(sr), up(w)
    k3.k3moe_combine(dims(d), od.data_ptr(), srd.data_ptr(), wd.data_ptr(), T, c.data_ptr(), stream())
    torch.cuda.synchronize()
    got = bf16_np(c)
    want = oracle.bf16_to_f64(oracle.combine(o.astype(np.float64), sr, w.astype(np.float64), T, d.top_k))
    o64, w64 = o.astype(np.float64), w.astype(np.float64)
    exact = np.stack([sum(w64[t, j] * o64[sr[t * d.top_k + j]] for j in range(d.top_k)) for t in range(T)])
    mag = np.stack([sum(abs(w64[t, j] * o64[sr[t * d.top_k + j]]) for j in range(d.top_k)) for t in range(T)])
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0**-8 + d.top_k * 2.0**-24 * mag * 1.01)
    assert rel_l2_rows(got, want).max() < 1e-3


# ------------------------------------------------------------------ whole layer
def _forward(lay, x_np, weights=None, dm=None):
    return run_layer(lay, x_np, weights, dm)


def _compare_layer(lay, x, y, idx, sample):
    return compare_layer(lay, x, y, idx, sample, nthreads=NCPU)


@pytest.mark.parametrize("actq", [0, 1])
def test_layer_tiny_every_token(actq):
    d = synth.TINY
    lay = DeviceLayer(d, seed=0, actq=actq)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y, idx, w = _forward(lay, x)
    err, flips = _compare_layer(lay, x, y, idx, np.arange(x.shape[0]))
    assert flips == 0


@pytest.mark.parametrize("actq", [0, 1])
def test_layer_tiny_prefill_every_token(actq):
    """150 tokens: tensor-core dense projections and block-scaled expert GEMMs."""
    d = synth.TINY
    lay = DeviceLayer(d, seed=2, actq=actq)
    T = 150
    x = synth.host_bf16_normal(11, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    y, idx, w = _forward(lay, x)
    _compare_layer(lay, x, y, idx, np.arange(T))


@pytest.mark.parametrize("T", [1, 3, 40, 150])  # routing: one block, a few blocks, one permutation block, many
def test_layer_stats_match_selection(T):
    d = synth.TINY
    lay = DeviceLayer(d, seed=6)
    x = synth.host_bf16_normal(8, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    dm = lay.dims
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=DEV)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
    ws, n = workspace(dm, T)
    xd = up(x)
    k3.k3moe_layer_forward(dm, lay.weights, xd.data_ptr(), T, y.data_ptr(), idx.data_ptr(), None, ws.data_ptr(),
                           n, stream())
    D, nbytes = k3.k3moe_layer_stats(dm, T, ws.data_ptr(), n, stream())
    check_ok(ws)
    want = len(np.unique(idx.cpu().numpy()))
    assert D == want
    assert nbytes == want * d.expert_bytes


@pytest.mark.parametrize("T", [1, 150])
def test_layer_in_cuda_graph_matches_direct_call(T):
    """The layer call neither allocates nor synchronises: captured in a CUDA graph and replayed,
    it gives the same bits as a direct call (two different token sets, replayed twice)."""
    d = synth.TINY
    lay = DeviceLayer(d, seed=7, shared=(2, 64))
    dm = lay.dims
    xs = [up(synth.host_bf16_normal(20 + i, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)) for i in range(2)]
    ys = [torch.empty((T, d.hidden), dtype=torch.int16, device=DEV) for _ in range(2)]
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
    ws, n = workspace(dm, T)
    direct = []
    for i in range(2):
        k3.k3moe_layer_forward(dm, lay.weights, xs[i].data_ptr(), T, ys[i].data_ptr(), idx.data_ptr(), None,
                               ws.data_ptr(), n, stream())
        direct.append(ys[i].clone())
    check_ok(ws)
    for yy in ys:
        yy.zero_()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        for i in range(2):
            k3.k3moe_layer_forward(dm, lay.weights, xs[i].data_ptr(), T, ys[i].data_ptr(), idx.data_ptr(), None,
                                   ws.data_ptr(), n, cs.cuda_stream)
    torch.cuda.current_stream().wait_stream(cs)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    check_ok(ws)
    for i in range(2):
        assert torch.equal(ys[i], direct[i])


def test_bounded_wait_runs_out_and_the_context_survives():
    """Failure detection without a fault: a device wait that nothing completes runs out after its
    wall-clock limit, the error word says so, and the next layer call runs and checks clean."""
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    k3.k3moe_selftest_timeout(ws.data_ptr(), stream())
    assert k3.k3moe_check(ws.data_ptr(), stream()) == 7  # K3MOE_E_TIMEOUT
    assert k3.k3moe_check(ws.data_ptr(), stream()) == k3.K3MOE_OK  # the word was cleared
    d = synth.TINY
    lay = DeviceLayer(d, seed=0)
    x = synth.host_x(synth.WORKLOADS["tiny"])
    y, idx, w = _forward(lay, x)  # checks the workspace error word itself
    _compare_layer(lay, x, y, idx, np.arange(x.shape[0]))


@pytest.mark.parametrize("T", [1, 64])
def test_decode_layer_completes_while_other_work_holds_most_sms(k3_layer, T):
    """The decode expert kernel's down items wait for GLU items of other CTAs. Its CTAs claim
    items from a counter, so the CTAs that are running do all the work even when other work
    keeps most SMs for longer than the device-side wait limit (2 s): here a finite load on a
    second stream holds all but 24 SMs for 3 s. The layer must finish clean, with the same bits
    as without the load."""
    x = synth.host_x(synth.WORKLOADS["decode_b64"], 0, T)
    want = _forward(k3_layer, x)
    n_sm = torch.cuda.get_device_properties(DEV).multi_processor_count
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    k3.k3moe_selftest_occupy(n_sm - 24, 3000, side.cuda_stream)
    time.sleep(0.3)  # the load has taken its SMs
    with torch.cuda.stream(main):
        got = _forward(k3_layer, x)  # checks the workspace error word (no timeout)
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_workspace_shared_across_token_counts(k3_layer):
    """One workspace, zeroed once, serves calls with different token counts in any order (the
    routing kernels' block counter sits in the fixed header): same bits as fresh workspaces."""
    x = synth.host_x(synth.WORKLOADS["decode_b64"], 0, 64)
    ws = workspace(k3_layer.dims, 64)
    for T in (1, 16, 3, 64, 2, 40, 1):
        got = run_layer(k3_layer, x[:T], ws=ws)
        want = run_layer(k3_layer, x[:T])
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)


def test_layer_tiny_ragged_and_edge_T():
    d = synth.TINY
    lay = DeviceLayer(d, seed=1, bias=synth.host_f32_normal(1, synth.S_BIAS, 0, d.n_experts, 1.0))
    for T in (1, 3, 9, 70, 193):
        x = synth.host_bf16_normal(T, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
        y, idx, w = _forward(lay, x)
        _compare_layer(lay, x, y, idx, np.arange(T))
    # T = 0 is a no-op
    dm = lay.dims
    ws, n = workspace(dm, 0)
    assert k3.k3moe_layer_forward(dm, lay.weights, 0, 0, 0, None, None, ws.data_ptr(), n, stream(),
                                  check=False) in (k3.K3MOE_OK, 1)


# Whole layer on shapes other than the tiny one: DEEP (several K stages per expert item, fewer
# items than SMs), HIDE (a residual wider than the latent, 64 experts) and ODD.
# ODD: latent and inter not multiples of 128 (the expert GEMV, the f16 block-scaled copy of z,
# and a last 128-row tile of W_in that is partly past its end).
HIDE = synth.Dims(hidden=1536, latent=512, inter=256, n_experts=64, top_k=4)
ODD = synth.Dims(hidden=256, latent=192, inter=192, n_experts=16, top_k=4)


@pytest.mark.parametrize("dname,T,actq", [("deep", 1, 0), ("deep", 5, 0), ("deep", 40, 0), ("hide", 1, 0),
                                          ("hide", 9, 0), ("hide", 64, 0), ("odd", 3, 0), ("odd", 70, 0),
                                          ("odd", 300, 0), ("wide", 7, 2), ("wide", 80, 2), ("deep", 5, 2),
                                          ("deep", 40, 2), ("hide", 64, 2), ("hide", 150, 2)])
def test_layer_other_dims_every_token(dname, T, actq):
    d = {"deep": DEEP, "hide": HIDE, "odd": ODD, "wide": WIDE}[dname]
    lay = DeviceLayer(d, seed=4, actq=actq)
    x = synth.host_bf16_normal(5, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    y, idx, w = _forward(lay, x)
    _compare_layer(lay, x, y, idx, np.arange(T))
    y2, idx2, w2 = _forward(lay, x)  # a rerun gives the same bits
    np.testing.assert_array_equal(y2, y)
    np.testing.assert_array_equal(idx2, idx)


# Two always-on shared experts beside the routed ones (width 64 on the tiny shape, 3072 on K3).
# With W_out = 0 the output is the shared experts' alone, y = bf16(s); otherwise
# y = bf16(W_out c + s). T = 3 runs the token-at-a-time projections, T = 150 the tensor-core ones.
@pytest.mark.parametrize("T", [3, 150])
@pytest.mark.parametrize("zero_out,actq", [(True, 0), (False, 0), (False, 1)])
def test_layer_shared_experts_every_token(T, zero_out, actq):
    d = synth.TINY
    lay = DeviceLayer(d, seed=3, shared=(2, 64), zero_out=zero_out, actq=actq)
    x = synth.host_bf16_normal(9, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    y, idx, w = _forward(lay, x)
    _compare_layer(lay, x, y, idx, np.arange(T))
    if zero_out:
        assert np.count_nonzero(y) > 0.9 * y.size


@pytest.mark.parametrize("T,sample", [(1, [0]), (64, [0, 31, 63]), (300, [0, 150, 299])])
def test_layer_k3_shared_experts_alone(T, sample):
    """K3 shapes, two shared experts of width 3072, W_out = 0: y = bf16(s) on sampled tokens."""
    d = synth.K3
    lay = DeviceLayer(d, seed=1, shared=(2, 3072), zero_out=True)
    try:
        x = synth.host_bf16_normal(12, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
        y, idx, w = _forward(lay, x)
        ol = lay.oracle(experts=[])
        for t in sample:
            s, _ = ol.shared_ffn(x[t])
            want = oracle.bf16_to_f64(oracle.bf16_from_f64(s))
            err = rel_l2_rows(y[t], want)
            assert err <= REL_L2, (t, err)
    finally:
        del lay
        torch.cuda.empty_cache()


@pytest.mark.parametrize("actq", [0, 1, 2])
def test_layer_k3_decode_b1(k3_layer, actq):
    w = synth.WORKLOADS["decode_b1"]
    n = 8
    x = synth.host_x(w, 0, n)
    dm = dims(k3_layer.d, actq)
    ys, idxs = [], []
    for t in range(n):  # one token per call, as in decode
        y, idx, _ = _forward(k3_layer, x[t:t + 1], dm=dm)
        ys.append(y[0])
        idxs.append(idx[0])
    k3_layer.actq = actq
    try:
        _compare_layer(k3_layer, x, np.stack(ys), np.stack(idxs), np.arange(n))
    finally:
        k3_layer.actq = 0


@pytest.mark.parametrize("actq", [0, 1, 2])
def test_layer_k3_decode_b64_biased(k3_layer, actq):
    w = synth.WORKLOADS["decode_b64"]
    bias = synth.router_bias(w)
    b = up(bias)
    lw = k3.Weights(*[getattr(k3_layer.weights, f) for f, _ in k3.Weights._fields_])
    lw.router_bias = b.data_ptr()
    k3_layer.bias_host = bias
    k3_layer.actq = actq
    try:
        x = synth.host_x(w)
        y, idx, _ = _forward(k3_layer, x, weights=lw, dm=dims(k3_layer.d, actq))
        distinct = len(np.unique(idx))
        assert distinct < 64 * 16  # reuse across the batch
        _compare_layer(k3_layer, x, y, idx, np.arange(64))  # every token of the step
    finally:
        k3_layer.bias_host = None
        k3_layer.actq = 0


def test_layer_k3_prefill_sampled(k3_layer):
    w = synth.WORKLOADS["prefill_4k"]
    T = 1024  # several chunks per expert, skewed routing
    bias = synth.router_bias(w)
    b = up(bias)
    lw = k3.Weights(*[getattr(k3_layer.weights, f) for f, _ in k3.Weights._fields_])
    lw.router_bias = b.data_ptr()
    k3_layer.bias_host = bias
    try:
        x = synth.host_x(w, 0, T)
        y, idx, _ = _forward(k3_layer, x, weights=lw)
        _compare_layer(k3_layer, x, y, idx, np.arange(0, T, 16))
    finally:
        k3_layer.bias_host = None


def _run_prepared(lay, h, x_np, ws):
    d = lay.d
    T = x_np.shape[0]
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=DEV)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, d.top_k), dtype=torch.float32, device=DEV)
    xd = up(x_np)
    k3.k3moe_layer_run(h, xd.data_ptr(), T, y.data_ptr(), idx.data_ptr(), w.data_ptr(), ws[0].data_ptr(), ws[1],
                       stream())
    check_ok(ws[0])
    return bf16_np(y), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,actq,Ts", [("tiny", 0, (1, 5, 8)), ("tiny", 1, (1, 8)), ("wide", 0, (1, 4)),
                                          ("deep", 1, (2, 80)), ("k3", 0, (1, 3, 64, 200)), ("k3", 1, (1, 16, 100)),
                                          ("k3", 2, (1, 70))])
def test_prepared_layer_same_bits_as_forward(name, actq, Ts, k3_layer):
    """k3moe_layer_run on a prepared layer (scales repacked once into the tensor-memory staging
    image) gives the bits k3moe_layer_forward gives: a misplaced scale would change them, since
    every expert's scales vary. tiny and wide cover stages of one 128-code chunk and a single
    two-chunk stage; K3 the full decode kernel; 70 tokens and more the many-token kernels, which
    take the GLU tile's interleaved image and the down image."""
    d = {"tiny": synth.TINY, "wide": WIDE, "deep": DEEP, "k3": synth.K3}[name]
    lay = k3_layer if name == "k3" else DeviceLayer(d, seed=3, actq=actq)
    dm = dims(d, actq=actq)  # (the weights do not depend on the activation mode)
    h = k3.k3moe_layer_init(dm, lay.weights, stream())
    try:
        for T in Ts:
            x = synth.host_x(synth.WORKLOADS["decode_b1"], 11, T) if name == "k3" else \
                synth.host_bf16_normal(9, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
            ws = workspace(dm, T)
            want = run_layer(lay, x, dm=dm, ws=ws)
            got = _run_prepared(lay, h, x, ws)
            for a, b in zip(got, want):
                np.testing.assert_array_equal(a, b)
    finally:
        k3.k3moe_layer_free(h)


# Many tokens with e4m3 activations: the experts with at most 8 rows run on the weights-on-N
# kernel and the others on the many-token kernel (chunks of 112 rows; 224 with MXFP8). A Zipf bias over
# WIDE's 16 experts gives both kinds, with counts on either side of the threshold (7, 8 / 9, 11
# at T = 96; 8 / 9, 13 and experts of more than one 112-row chunk at T = 200). Every token is
# compared with the oracle, and the prepared layer (scales from the packed images) gives the
# same bits as the unprepared one. With MXFP4 activations (no small-expert kernel) the 200-row
# experts fill a 192-row chunk, whose activation rows 128.. take the second block of scales.
@pytest.mark.parametrize("wseed,bseed,T,actq", [(3, 3, 96, 0), (7, 4, 200, 0), (7, 4, 200, 1), (7, 4, 200, 2)])
def test_layer_small_and_large_experts(wseed, bseed, T, actq):
    d = WIDE
    lay = DeviceLayer(d, seed=wseed, bias=synth.zipf_bias(d.n_experts, bseed, s=0.7), actq=actq)
    x = synth.host_bf16_normal(5, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
    y, idx, w = _forward(lay, x)
    cnt = np.bincount(idx.ravel(), minlength=d.n_experts)
    assert ((cnt > 0) & (cnt <= 8)).sum() >= 2 and (cnt > 8).sum() >= 3, sorted(cnt.tolist())
    _compare_layer(lay, x, y, idx, np.arange(T))
    dm = dims(d, actq=actq)
    h = k3.k3moe_layer_init(dm, lay.weights, stream())
    try:
        ws = workspace(dm, T)
        want = run_layer(lay, x, dm=dm, ws=ws)
        got = _run_prepared(lay, h, x, ws)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)
    finally:
        k3.k3moe_layer_free(h)


@pytest.mark.parametrize("name,Ts", [("tiny", (1, 8, 100)), ("k3", (1, 64))])
def test_layer_run_host_same_bits(name, Ts, k3_layer):
    """k3moe_layer_run_host (tokens read from and output written to page-locked host memory by
    the library's own copy kernels) gives the bits k3moe_layer_run gives; a pageable buffer is
    refused with K3MOE_E_HOSTMEM before anything is launched."""
    d = {"tiny": synth.TINY, "k3": synth.K3}[name]
    lay = k3_layer if name == "k3" else DeviceLayer(d, seed=3)
    dm = dims(d)
    h = k3.k3moe_layer_init(dm, lay.weights, stream())
    try:
        for T in Ts:
            x = synth.host_bf16_normal(13, synth.S_X, 0, T * d.hidden, 1.0).reshape(T, d.hidden)
            ws = workspace(dm, T)
            want = _run_prepared(lay, h, x, ws)
            xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
            yh = torch.full((T, d.hidden), -1, dtype=torch.int16).pin_memory()
            idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
            w = torch.empty((T, d.top_k), dtype=torch.float32, device=DEV)
            k3.k3moe_layer_run_host(h, xh.data_ptr(), T, yh.data_ptr(), idx.data_ptr(), w.data_ptr(),
                                    ws[0].data_ptr(), ws[1], stream())
            check_ok(ws[0])
            np.testing.assert_array_equal(bf16_np(yh), want[0])
            np.testing.assert_array_equal(idx.cpu().numpy(), want[1])
            np.testing.assert_array_equal(w.cpu().numpy(), want[2])
            pageable = np.zeros((T, d.hidden), np.int16)
            st = k3.k3moe_layer_run_host(h, pageable.ctypes.data, T, yh.data_ptr(), None, None, ws[0].data_ptr(),
                                         ws[1], stream(), check=False)
            assert st == 10, k3.status_string(st)
    finally:
        k3.k3moe_layer_free(h)
