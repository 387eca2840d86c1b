"""Stage-by-stage parity of the layer at K3 size, each stage fed the oracle's own input (never
a GPU value into the oracle): where the GPU's bf16 results differ from the oracle's, the
difference is a rounding straddle of an fp32 sum.

- z = bf16(W_in x) (k3moe_project, token-at-a-time and tensor-core paths): every element that
  differs is the neighbouring bf16 value, with the exact sum within an fp32 error bound of
  the midpoint between the two.
- Expert rows on the oracle's z (k3moe_expert_ffn_mxfp4, both expert kernels): each row within
  2e-3, most within a few fp32 ulps (the rest carry a straddle of one GLU output element).
- y = bf16(W_out c) on the oracle's c: straddles only, as for z."""
import os

import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth
from k3help import (DEV, REL_L2, DeviceLayer, up, stream, workspace, check_ok, rel_l2_rows,
                    check_rounding_straddles)

pytestmark = pytest.mark.gpu
NCPU = os.cpu_count() or 8
f64 = oracle.bf16_to_f64


@pytest.fixture(scope="module")
def lay():
    w = synth.WORKLOADS["prefill_4k"]
    lay = DeviceLayer(synth.K3, seed=0, bias=synth.router_bias(w))
    torch.cuda.synchronize()
    yield lay
    del lay
    torch.cuda.empty_cache()


def _project(W, x, N, K):
    T = x.shape[0]
    out = torch.empty((T, N), dtype=torch.int16, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    Wd, xd = up(W), up(x)
    k3.k3moe_project(Wd.data_ptr(), xd.data_ptr(), T, N, K, out.data_ptr(), ws.data_ptr(), 256, stream())
    check_ok(ws)
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T", [1, 32, 64, 2048])  # 1, 32: token-at-a-time kernel; 64, 2048: tensor cores
def test_latent_in_differs_only_by_rounding_straddles(lay, T):
    d = lay.d
    x = synth.host_x(synth.WORKLOADS["prefill_4k"], 0, T)
    wi = lay.dense()[1]
    z = _project(wi, x, d.latent, d.hidden)
    xf, wf = f64(x), f64(wi)
    exact = xf @ wf.T
    mag = np.abs(xf) @ np.abs(wf).T
    flips = check_rounding_straddles(z, exact, mag)
    print(f"z, {T} tokens: straddles per token mean {flips.mean():.2f} max {flips.max()}")
    assert flips.max() <= 12


@pytest.mark.parametrize("T,reps", [(16, 1), (16, 5)])  # 16 tokens: decode kernel; 80: many-token kernel
def test_expert_rows_on_the_oracles_z(lay, T, reps):
    d = lay.d
    x = synth.host_x(synth.WORKLOADS["prefill_4k"], 0, T)
    sel = oracle.select_topk(oracle.router_logits_np(x, lay.dense()[0], lay.bias_host), d.top_k)
    ol = lay.oracle(experts=set(sel.ravel().tolist()))
    ref = ol.forward_np(x, nthreads=NCPU)
    z, idx = np.concatenate([ref["z"]] * reps), np.concatenate([ref["idx"]] * reps)
    Tr = z.shape[0]
    off, rt, rs, sr = oracle.permute(idx, d.n_experts)
    o = torch.empty((Tr * d.top_k, d.latent), dtype=torch.float32, device=DEV)
    ws, n = workspace(lay.dims, Tr)
    zd, offd, rtd = up(z), up(off), up(rt)
    k3.k3moe_expert_ffn_mxfp4(lay.dims, lay.weights, zd.data_ptr(), Tr, offd.data_ptr(), rtd.data_ptr(),
                              o.data_ptr(), ws.data_ptr(), n, stream())
    check_ok(ws)
    o = o.cpu().numpy().astype(np.float64)
    got = np.stack([o[sr[t * d.top_k + j]] for t in range(T) for j in range(d.top_k)])
    want = ref["o"].reshape(T * d.top_k, d.latent)
    err = rel_l2_rows(got, want)
    print(f"expert rows on the oracle's z ({Tr} tokens): median {np.median(err):.2e}, max {err.max():.2e}, "
          f"{int((err > 1e-5).sum())} of {len(err)} rows above 1e-5")
    assert err.max() <= REL_L2
    assert np.median(err) <= 2e-6
    assert (err > 1e-5).mean() <= 0.3


def test_latent_out_on_the_oracles_c_differs_only_by_rounding_straddles(lay):
    d = lay.d
    x = synth.host_x(synth.WORKLOADS["prefill_4k"], 0, 16)
    sel = oracle.select_topk(oracle.router_logits_np(x, lay.dense()[0], lay.bias_host), d.top_k)
    ref = lay.oracle(experts=set(sel.ravel().tolist())).forward_np(x, nthreads=NCPU)
    wo = lay.dense()[2]
    y = _project(wo, ref["c"], d.hidden, d.latent)
    cf, wf = f64(ref["c"]), f64(wo)
    flips = check_rounding_straddles(y, cf @ wf.T, np.abs(cf) @ np.abs(wf).T)
    print(f"y on the oracle's c: straddles per token mean {flips.mean():.2f} max {flips.max()}")
    np.testing.assert_array_equal(y[flips == 0], ref["y"][flips == 0])
