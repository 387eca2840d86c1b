"""k3moe_route_noalloc against k3moe_route, through the C ABI, on the GPU.

k3moe_route_noalloc serves callers that may not allocate device memory at all, for instance a
serving process whose device memory belongs to its own pool allocator and which keeps
cudaMalloc / cudaFree off the request path because those calls can synchronise the whole
device. It keeps the router logits in a fixed scratch array inside the library instead of a
caller workspace. This file is named to be collected last, so a run that stops at the first
failure has run every other test before this one; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth
from k3help import DEV, LOGIT_RTOL, boundary_tol, selection_valid, stream, topk_gap_ambiguous, up

pytestmark = pytest.mark.gpu

# K3 router widths: 7168-wide tokens, 896 experts, top-16
H, E, K = 7168, 896, 16


def _dims():
    return k3.Dims(H, 3584, 3072, E, K, 0, 0)


def _route_with_workspace(dm, xd, T, wd, bd):
    idx = torch.empty((T, K), dtype=torch.int32, device=DEV)
    w = torch.empty((T, K), dtype=torch.float32, device=DEV)
    n = k3.k3moe_workspace_size(dm, T)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    k3.k3moe_route(dm, xd.data_ptr(), T, wd.data_ptr(), bd.data_ptr() if bd is not None else None, None,
                   idx.data_ptr(), w.data_ptr(), ws.data_ptr(), n, stream())
    assert k3.k3moe_check(ws.data_ptr(), stream()) == k3.K3MOE_OK
    return idx.cpu().numpy(), w.cpu().numpy()


def _route_no_alloc(dm, xd, T, wd, bd, err):
    idx = torch.full((T, K), -7, dtype=torch.int32, device=DEV)
    w = torch.full((T, K), -7.0, dtype=torch.float32, device=DEV)
    k3.k3moe_route_noalloc(dm, xd.data_ptr(), T, wd.data_ptr(), bd.data_ptr() if bd is not None else None,
                           idx.data_ptr(), w.data_ptr(), err.data_ptr() if err is not None else None, stream())
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def test_route_noalloc_matches_route_on_consecutive_calls():
    dm = _dims()
    wr = synth.host_bf16_normal(0, synth.S_W_ROUTER, 0, E * H, 0.02).reshape(E, H)
    bias = synth.host_f32_normal(0, synth.S_BIAS, 0, E, 1.0).astype(np.float32)
    wd, bd = up(wr), up(bias)
    err = torch.full((1,), 0xFFFF, dtype=torch.int32, device=DEV)  # must come back cleared
    # two calls in a row with different token counts and inputs: the second runs on the scratch
    # the first left behind; then a call without an error word
    for call, (T, seed, b) in enumerate([(64, 1, bd), (5, 2, None), (73, 3, bd)]):
        x = synth.host_bf16_normal(seed, synth.S_X, 0, T * H, 1.0).reshape(T, H)
        xd = up(x)
        want_idx, want_w = _route_with_workspace(dm, xd, T, wd, b)
        got_idx, got_w = _route_no_alloc(dm, xd, T, wd, b, err if call < 2 else None)
        np.testing.assert_array_equal(got_idx, want_idx)
        np.testing.assert_allclose(got_w, want_w, rtol=LOGIT_RTOL, atol=0)
        if call < 2:
            assert int(err.item()) == 0
        # and against the oracle (double logits, brute-force top-k): bit-exact except tokens
        # whose k-th and (k+1)-th logits tie within the fp32 error, which must select validly
        ref_lg = oracle.router_logits_np(x, wr, None if b is None else bias)
        ref_idx = oracle.select_topk(ref_lg, K)
        tol = boundary_tol(ref_lg)
        same = np.all(got_idx == ref_idx, axis=1)
        assert np.all(same | topk_gap_ambiguous(ref_lg, K, tol))
        for t in np.nonzero(~same)[0]:
            assert selection_valid(ref_lg[t], got_idx[t], K, 2 * tol[t])
        np.testing.assert_allclose(got_w[same], oracle.route_weights(ref_lg, ref_idx)[same], rtol=5e-4, atol=1e-6)


def test_route_noalloc_rejects_requests_beyond_its_scratch():
    dm = _dims()
    good = 1 << 16  # never dereferenced: the checks come before any launch
    st = k3.k3moe_route_noalloc(dm, good, 74, good, None, good, good, None, stream(), check=False)
    assert st == 9 and k3.status_string(st).startswith("K3MOE_E_SCRATCH")
    assert k3.k3moe_route_noalloc(dm, None, 4, good, None, good, good, None, stream(), check=False) == 1
    assert k3.k3moe_route_noalloc(dm, good + 2, 4, good, None, good, good, None, stream(), check=False) == 3
    assert k3.k3moe_route_noalloc(dm, good, 0, good, None, good, good, None, stream()) == k3.K3MOE_OK
