"""REAP saliency accumulation and the per-expert cosine verifier, on the GPU against the oracle.

"kimi-k3-mlx" digest:
- REAP pruning section: expert j's saliency S_j = (1/|C|) sum_x g_j(x) ||e_j(x)||_2.
  k3moe_layer_saliency accumulates the step's sums of g * ||o|| per expert; the test
  compares them with the oracle's over the same tokens, across several layer calls on both
  expert paths.
- verify.py paragraph: a per-expert cosine similarity between two computations of each
  expert, which quantisation noise barely moves but which a mis-stacked expert or a
  transposed matrix drops to about 0. Here: the GPU's expert rows against the oracle's on probe
  rows, for every expert of a K3 layer. The planted mistakes sit in the oracle's copy of the
  experts (on the CPU)."""
import os

import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth
from k3help import DEV, DeviceLayer, up, stream, workspace, check_ok, check_selection

pytestmark = pytest.mark.gpu
NCPU = os.cpu_count() or 8


@pytest.fixture(scope="module")
def lay():
    w = synth.WORKLOADS["prefill_4k"]
    lay = DeviceLayer(synth.K3, seed=0, bias=synth.router_bias(w))
    torch.cuda.synchronize()
    yield lay
    del lay
    torch.cuda.empty_cache()


def test_layer_saliency_matches_the_oracle(lay):
    d = lay.d
    x = synth.host_x(synth.WORKLOADS["prefill_4k"], 0, 512)
    S = torch.zeros(d.n_experts, dtype=torch.float64, device=DEV)
    idx_all = []
    # calls of 1, 16, 64 (decode expert kernel) and 431 tokens (many-token kernel), one workspace
    wsb, n = workspace(lay.dims, 431)
    for call, (a, b) in enumerate(((0, 1), (1, 17), (17, 81), (81, 512))):
        T = b - a
        xd = up(x[a:b])
        y = torch.empty((T, d.hidden), dtype=torch.int16, device=DEV)
        if call % 2 == 0:  # the routing through the call's outputs
            idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
            wt = torch.empty((T, d.top_k), dtype=torch.float32, device=DEV)
            ip, wp = idx.data_ptr(), wt.data_ptr()
        else:  # ... or kept in the workspace (NULL outputs)
            ip = wp = None
        k3.k3moe_layer_forward(lay.dims, lay.weights, xd.data_ptr(), T, y.data_ptr(), ip, wp, wsb.data_ptr(), n,
                               stream())
        k3.k3moe_layer_saliency(lay.dims, T, ip, wp, wsb.data_ptr(), n, S.data_ptr(), stream())
        check_ok(wsb)
        if ip is None:  # the selection of this call, for the oracle: route the same tokens again
            idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
            k3.k3moe_layer_forward(lay.dims, lay.weights, xd.data_ptr(), T, y.data_ptr(), idx.data_ptr(), None,
                                   wsb.data_ptr(), n, stream())
            check_ok(wsb)
        idx_all.append(idx.cpu().numpy())
    gidx = np.concatenate(idx_all)
    check_selection(lay, x, gidx)
    ol = lay.oracle(experts=set())
    ref = ol.forward_with_selection(x, gidx, nthreads=2 * NCPU, rows_fn=lay.rows_fn())
    want = oracle.saliency_accumulate(d, ref["idx"], ref["w"], ref["o"])
    got = S.cpu().numpy()
    used = want > 0
    assert np.array_equal(got > 0, used)
    rel = np.abs(got[used] - want[used]) / want[used]
    print(f"saliency: {int(used.sum())} experts, max relative error {rel.max():.2e}")
    assert rel.max() <= 1e-4


def _probe_selection(experts, k, reps=2):
    """Tokens whose k slots cover every listed expert reps times (distinct experts per token)."""
    ex = list(experts) * reps
    T = (len(ex) + k - 1) // k
    ex += list(experts)[: T * k - len(ex)]
    idx = np.array(ex, np.int32).reshape(T, k)
    return np.sort(idx, axis=1)


def expert_cosines(lay, experts, oracle_rows, seed=3):
    """The verifier: per expert, cosine similarity between the GPU's expert rows
    (k3moe_expert_ffn_mxfp4) and oracle_rows(e, z_rows) on the same probe z rows."""
    d = lay.d
    idx = _probe_selection(experts, d.top_k)
    T = idx.shape[0]
    z = synth.host_bf16_normal(seed, synth.S_X, 0, T * d.latent, 1.7).reshape(T, d.latent)
    off, rt, rs, sr = oracle.permute(idx, d.n_experts)
    o = torch.empty((T * d.top_k, d.latent), dtype=torch.float32, device=DEV)
    ws, n = workspace(lay.dims, T)
    zd, offd, rtd = up(z), up(off), up(rt)
    k3.k3moe_expert_ffn_mxfp4(lay.dims, lay.weights, zd.data_ptr(), T, offd.data_ptr(), rtd.data_ptr(), o.data_ptr(),
                              ws.data_ptr(), n, stream())
    check_ok(ws)
    o = o.cpu().numpy().astype(np.float64)
    cos = {}
    for e in experts:
        t, j = np.nonzero(idx == e)
        g = np.stack([o[sr[a * d.top_k + b]] for a, b in zip(t, j)])
        w = oracle_rows(int(e), z[t])
        cos[int(e)] = float(np.sum(g * w) / (np.linalg.norm(g) * np.linalg.norm(w)))
    return cos


def test_verifier_every_expert_of_a_k3_layer(lay):
    from concurrent.futures import ThreadPoolExecutor
    import oracle_pool
    rf = oracle_pool.rows_fn(lay.d, lay.seed, 0)
    experts = list(range(lay.d.n_experts))
    cache = {}

    def rows(e, zr):
        return cache[e]

    # oracle rows of all experts, in parallel, then the cosines
    idx = _probe_selection(experts, lay.d.top_k)
    z = synth.host_bf16_normal(3, synth.S_X, 0, idx.shape[0] * lay.d.latent, 1.7).reshape(idx.shape[0], -1)
    with ThreadPoolExecutor(2 * NCPU) as pool:
        for e, r in zip(experts, pool.map(lambda e: rf(e, z[np.nonzero(idx == e)[0]]), experts)):
            cache[e] = r
    cos = expert_cosines(lay, experts, rows)
    worst = min(cos.values())
    print(f"verifier: {len(cos)} experts, lowest cosine 1 - {1 - worst:.2e}")
    assert worst >= 1 - 1e-6


@pytest.mark.parametrize("mistake", ["mis-stacked", "transposed"])
def test_verifier_flags_a_planted_mistake(mistake):
    """The oracle's copy of expert 3 carries the mistake: expert 4's tensors in its place
    (mis-stacked), or its down matrix transposed (the tiny layer's down matrix is square). Its
    cosine falls near 0; every other expert stays at 1."""
    d = synth.TINY
    lay = DeviceLayer(d, seed=0)
    ex = {e: dict(synth.host_expert(d, 0, e)) for e in range(d.n_experts)}
    if mistake == "mis-stacked":
        ex[3] = dict(ex[4])
    else:
        q = ex[3]["down_q"]
        codes = np.empty((d.latent, d.inter), np.uint8)
        codes[:, 0::2], codes[:, 1::2] = q & 0xF, q >> 4
        ct = codes.T.copy()
        ex[3]["down_q"] = (ct[:, 0::2] | (ct[:, 1::2] << 4)).astype(np.uint8)
        ex[3]["down_s"] = ex[3]["down_s"].copy()  # same scales, now misapplied along the other axis
    wr, wi, wo = synth.host_dense(d, 0)
    bad = oracle.Layer(d, wr, wi, wo, ex)
    cos = expert_cosines(lay, range(d.n_experts), lambda e, zr: oracle.expert_rows(d, bad.experts[e], zr))
    print(f"verifier, {mistake} expert 3: cosine {cos[3]:.3f}; others >= {min(v for e, v in cos.items() if e != 3):.6f}")
    assert abs(cos[3]) < 0.3
    assert all(v >= 1 - 1e-6 for e, v in cos.items() if e != 3)
