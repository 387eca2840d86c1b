"""Shared helpers of the GPU tests: device layers filled by the seeded generator, the matching
oracle layer built from host-generated tensors, and comparison rules.

Inputs reach the oracle only from the host generator (synth, host side) and reach the GPU
from the device generator or a host->device copy of the same host arrays; nothing the CUDA
library computes is fed to the oracle.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth

DEV = torch.device("cuda:0")
NAMES = oracle.ExpertTables.NAMES

# Tolerances. Indices and permutations: bit-exact. Layer outputs against the oracle:
# - bf16 activations: the relative L2 error of the compared output (all compared tokens
#   together) within REL_L2 = 2e-3; every token within PER_TOKEN_CAP[0], and above REL_L2 on at
#   most PER_TOKEN_OVER_FRAC[0] of the tokens when 32 or more are compared.
# - MXFP8 activations: every token within PER_TOKEN_CAP[1], above REL_L2 on at most
#   PER_TOKEN_OVER_FRAC[1] of the tokens (at most one token when fewer than 20 are compared), and
#   the compared output within REL_L2 when WHOLE_MIN_TOKENS[1] or more tokens are compared.
# Why a per-token envelope: the layer has four bf16 rounding points (z, the GLU output, the
# combine, y); an fp32 sum that lands across a bf16 rounding midpoint flips that element, and
# the flip perturbs every later rounding point. A plain fp32 evaluation of the layer on the CPU
# (fp32_layer.py) against the oracle shows this envelope (1024 K3 prefill tokens): bf16 mode
# whole 9.9e-4, per token max 2.9e-3 with 7% of the tokens above 2e-3; MXFP8 mode whole
# 1.5e-3, median 1.6e-6, 1.7% of the tokens above 2e-3 and a few near 1e-2 (max 2.2e-2): where
# a straddle of z falls on an E4M3 rounding midpoint the element moves by a whole E4M3 step.
# test_tolerance_reading.py re-runs the bf16 case as a CPU test. Narrow layers (latent < 1024,
# the small test shapes) have fewer elements per token, so one straddle weighs more: the same
# fp32 evaluation on 3000 tokens of each small test shape reaches 4.8e-3 per token in bf16 mode
# (1.7e-2 in MXFP8 mode), hence PER_TOKEN_CAP_NARROW.
# MXFP4 activations (actq 2; the target states no tolerance for this mode, so it is derived the
# same way): the e2m1 rounding points are coarser still. The fp32 evaluation on 512 tokens: median
# 5.9e-7, p99 5.5e-4, one token at 3.9e-2 (a straddle of z on an e2m1 boundary) that alone makes
# the whole-output error 1.4e-3; hence a per-token cap of 8e-2, at most 2% of the tokens above
# 2e-3, and the compared output within WHOLE_BOUND[2] over 1024 tokens or more.
REL_L2 = 2e-3
PER_TOKEN_CAP = {0: 4e-3, 1: 3e-2, 2: 8e-2}
PER_TOKEN_CAP_NARROW = {0: 6e-3, 1: 3e-2, 2: 8e-2}
PER_TOKEN_OVER_FRAC = {0: 0.2, 1: 0.05, 2: 0.02}
WHOLE_MIN_TOKENS = {0: 1, 1: 1024, 2: 1024}
WHOLE_BOUND = {0: REL_L2, 1: REL_L2, 2: 2 * REL_L2}
# Expert rows (one (token, expert) pair, fp32 out, no later rounding point): REL_L2 per row.
# fp32 logits against double logits: |dl| <= LOGIT_ATOL + LOGIT_RTOL * |l|
LOGIT_ATOL, LOGIT_RTOL = 1e-4, 1e-4


def stream():
    return torch.cuda.current_stream().cuda_stream


def up(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_to_f64(t.cpu().numpy().view(np.uint16))


def dims(d: synth.Dims, actq=0, act=0, shared=None) -> k3.Dims:
    ns, si = shared or (0, 0)
    return k3.Dims(d.hidden, d.latent, d.inter, d.n_experts, d.top_k, act, actq, ns, si)


class DeviceLayer:
    """A whole layer resident on the GPU. Small layers are generated on the host and copied;
    K3-sized ones are generated on the device (byte-identical generator)."""

    def __init__(self, d: synth.Dims, seed=0, bias=None, actq=0, host_fill=None, experts=None, shared=None,
                 zero_out=False):
        """shared: (n_shared, shared_inter) or None; zero_out: W_out = 0, so that y is the shared
        experts' output alone."""
        self.d, self.seed, self.actq, self.shared, self.zero_out = d, seed, actq, shared, zero_out
        E = d.n_experts
        if host_fill is None:
            host_fill = E * d.expert_bytes < 64 << 20
        self.host_fill = host_fill
        self._custom_experts = experts is not None
        self.t = {}
        if host_fill:
            wr, wi, wo = synth.host_dense(d, seed)
            self.dense_host = (wr, wi, wo)
            ex = experts if experts is not None else {e: synth.host_expert(d, seed, e) for e in range(E)}
            self._experts_host = ex
            self.t["w_router"], self.t["w_in"], self.t["w_out"] = up(wr), up(wi), up(wo)
            for n in NAMES:
                self.t[n] = up(np.stack([ex[e][n] for e in range(E)]))
        else:
            assert experts is None
            self.dense_host = None
            self._experts_host = {}
            sizes = {"w_router": E * d.hidden * 2, "w_in": d.latent * d.hidden * 2,
                     "w_out": d.hidden * d.latent * 2, "gate_q": E * d.gate_q_bytes,
                     "gate_s": E * d.gate_s_bytes, "up_q": E * d.gate_q_bytes,
                     "up_s": E * d.gate_s_bytes, "down_q": E * d.down_q_bytes,
                     "down_s": E * d.down_s_bytes}
            for n, b in sizes.items():
                self.t[n] = torch.empty(b, dtype=torch.uint8, device=DEV)
            synth.dev_fill_layer(d, seed, {n: v.data_ptr() for n, v in self.t.items()}, stream())
        if zero_out:
            self.t["w_out"].zero_()
        self.shared_host = None
        sp = [None, None, None]
        if shared is not None:
            ns, si = shared
            S = ns * si
            if host_fill:
                self.shared_host = synth.host_shared(d, ns, si, seed)
                for i, n in enumerate(("w_sgate", "w_sup", "w_sdown")):
                    self.t[n] = up(self.shared_host[i])
            else:
                for n in ("w_sgate", "w_sup", "w_sdown"):
                    self.t[n] = torch.empty(S * d.hidden * 2, dtype=torch.uint8, device=DEV)
                synth.dev_fill_shared(d, ns, si, seed, {n: self.t[n].data_ptr() for n in ("w_sgate", "w_sup", "w_sdown")},
                                      stream())
            sp = [self.t[n].data_ptr() for n in ("w_sgate", "w_sup", "w_sdown")]
        self.bias_host = None if bias is None else np.ascontiguousarray(bias, np.float32)
        self.t["bias"] = None if bias is None else up(self.bias_host)
        self.dims = dims(d, actq, shared=shared)
        self.weights = k3.Weights(self.t["w_router"].data_ptr(),
                                  None if bias is None else self.t["bias"].data_ptr(),
                                  self.t["w_in"].data_ptr(), self.t["w_out"].data_ptr(),
                                  *[self.t[n].data_ptr() for n in NAMES], *sp)

    def rows_fn(self, actq=None):
        """For K3-sized layers whose experts come from the seeded generator: the oracle's expert
        rows computed in a process pool (oracle_pool); else None (in process)."""
        if self.d.latent < 1024 or self.host_fill and self._custom_experts:
            return None
        import oracle_pool
        return oracle_pool.rows_fn(self.d, self.seed, self.actq if actq is None else actq)

    def dense(self):
        if self.dense_host is None:
            self.dense_host = synth.host_dense(self.d, self.seed)
        wr, wi, wo = self.dense_host
        return (wr, wi, np.zeros_like(wo)) if self.zero_out else (wr, wi, wo)

    def expert_host(self, e):
        if e not in self._experts_host:
            self._experts_host[e] = synth.host_expert(self.d, self.seed, e)
        return self._experts_host[e]

    def oracle(self, experts=None, actq=None):
        ids = [int(e) for e in (range(self.d.n_experts) if experts is None else experts)]
        missing = [e for e in ids if e not in self._experts_host]
        if len(missing) > 8:  # the host generator releases the GIL: fill them in parallel
            from concurrent.futures import ThreadPoolExecutor
            with ThreadPoolExecutor(os.cpu_count() or 8) as pool:
                for e, t in zip(missing, pool.map(lambda e: synth.host_expert(self.d, self.seed, e), missing)):
                    self._experts_host[e] = t
        ex = {e: self.expert_host(e) for e in ids}
        wr, wi, wo = self.dense()
        sh = None
        if self.shared is not None:
            if self.shared_host is None:
                self.shared_host = synth.host_shared(self.d, *self.shared, self.seed)
            sh = (*self.shared_host, self.shared[0])
        return oracle.Layer(self.d, wr, wi, wo, ex, bias=self.bias_host,
                            actq=self.actq if actq is None else actq, shared=sh)


def workspace(dm: k3.Dims, T: int) -> tuple[torch.Tensor, int]:
    n = k3.k3moe_workspace_size(dm, T)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=DEV), n


def check_ok(ws: torch.Tensor):
    st = k3.k3moe_check(ws.data_ptr(), stream())
    assert st == k3.K3MOE_OK, k3.status_string(st)


def rel_l2_rows(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    num = np.linalg.norm(got - want, axis=-1)
    den = np.linalg.norm(want, axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


def boundary_tol(logits: np.ndarray) -> np.ndarray:
    """Per token: twice the fp32 logit error bound at that token's own largest logit."""
    return 2 * (LOGIT_ATOL + LOGIT_RTOL * np.abs(logits).max(axis=1))


def topk_gap_ambiguous(logits: np.ndarray, k: int, tol: np.ndarray | float) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest oracle logits are closer than tol (per token or
    one value): there the selection at the boundary is decided below the precision of fp32
    logits."""
    srt = -np.sort(-logits, axis=1)
    if k >= logits.shape[1]:
        return np.zeros(logits.shape[0], bool)
    gap = srt[:, k - 1] - srt[:, k]
    return gap < tol


def selection_valid(logits_row: np.ndarray, sel: np.ndarray, k: int, tol: float) -> bool:
    """A selection is valid when no unselected logit beats a selected one by more than tol."""
    mask = np.zeros(logits_row.shape[0], bool)
    mask[sel] = True
    if len(set(sel.tolist())) != k:
        return False
    return logits_row[mask].min() >= logits_row[~mask].max() - tol


def check_layer_output(got: np.ndarray, want: np.ndarray, what: str = "layer", actq: int = 0,
                       latent: int = 3584) -> np.ndarray:
    """Layer outputs (rows = tokens, values as doubles) against the oracle's, by the rules above
    for the activation mode actq and the layer's latent width. Returns the per-token errors."""
    err = rel_l2_rows(got, want)
    whole = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    over = int((err > REL_L2).sum())
    n = len(err)
    print(f"{what}: rel L2 whole {whole:.3e}, per token median {np.median(err):.3e} max {err.max():.3e}, "
          f"{over} of {n} tokens above {REL_L2}")
    m = actq
    if n >= WHOLE_MIN_TOKENS[m]:
        assert whole <= WHOLE_BOUND[m], (what, whole)
    cap = (PER_TOKEN_CAP if latent >= 1024 else PER_TOKEN_CAP_NARROW)[m]
    assert err.max() <= cap, (what, err.max(), cap)
    if m == 0 and n >= 32:
        assert over <= PER_TOKEN_OVER_FRAC[0] * n, (what, over, n)
    if m != 0:
        assert over <= max(1, PER_TOKEN_OVER_FRAC[m] * n), (what, over, n)
    return err


def compare_layer(lay, x: np.ndarray, y: np.ndarray, idx: np.ndarray, sample, nthreads: int = 8,
                  what: str = "layer"):
    """The GPU's y and selection for the sampled tokens against the oracle.
    Selections: bit-exact, except on tokens whose k-th and (k+1)-th oracle logits are closer than
    the fp32 logit error (boundary ties), where the GPU's selection must be valid (no unselected
    logit above a selected one by more than the tolerance). Outputs: the oracle computes every
    token with its own selection, and each boundary-tie token whose selection differs a second
    time with the GPU's selection (the oracle completed with it); both go through
    check_layer_output. Returns (per-token errors, number of boundary-tie tokens)."""
    d = lay.d
    sample = np.asarray(sample)
    xs, gi = x[sample], idx[sample]
    rf = lay.rows_fn()
    ol = lay.oracle(experts=set() if rf else set(np.unique(gi).tolist()) | _own_selection(lay, xs))
    nthreads = 2 * nthreads if rf else nthreads
    ref = ol.forward_np(xs, nthreads=nthreads, rows_fn=rf)
    lg = ref["logits"]
    tol = boundary_tol(lg)
    amb = topk_gap_ambiguous(lg, d.top_k, tol)
    same = np.all(gi == ref["idx"], axis=1)
    assert np.all(same | amb), f"{int((~same & ~amb).sum())} tokens select other experts"
    want = ref["y"].copy()
    flipped = np.nonzero(~same)[0]
    for t in flipped:
        assert selection_valid(lg[t], gi[t], d.top_k, 2 * tol[t]), t
    if len(flipped):
        want[flipped] = ol.forward_with_selection(xs[flipped], gi[flipped], nthreads=nthreads, rows_fn=rf)["y"]
    err = check_layer_output(bf16_np_bits(y[sample]), oracle.bf16_to_f64(want), what, lay.actq, d.latent)
    return err, len(flipped)


def _own_selection(lay, xs) -> set:
    wr = lay.dense()[0]
    return set(oracle.select_topk(oracle.router_logits_np(xs, wr, lay.bias_host), lay.d.top_k).ravel().tolist())


def bf16_np_bits(a) -> np.ndarray:
    """bf16 values given as uint16 bits or as doubles already -> doubles."""
    a = np.asarray(a)
    return oracle.bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def run_layer(lay, x_np: np.ndarray, weights=None, dm=None, ws=None):
    """k3moe_layer_forward on x (host bf16 bits): (y as doubles, topk_idx, topk_w), with the
    workspace error word checked. ws: (tensor, bytes) to reuse, else one is allocated."""
    d = lay.d
    dm = dm or lay.dims
    T = x_np.shape[0]
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=DEV)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, d.top_k), dtype=torch.float32, device=DEV)
    wsb, n = ws if ws is not None else workspace(dm, T)
    xd = up(x_np)
    k3.k3moe_layer_forward(dm, weights or lay.weights, xd.data_ptr(), T, y.data_ptr(), idx.data_ptr(), w.data_ptr(),
                           wsb.data_ptr(), n, stream())
    check_ok(wsb)
    return bf16_np(y), idx.cpu().numpy(), w.cpu().numpy()


def check_selection(lay, x: np.ndarray, idx: np.ndarray) -> int:
    """The GPU's top-k of every token against the oracle's selection on double logits:
    bit-exact except boundary ties, where the selection must be valid. Returns the number of
    boundary-tie tokens that selected differently."""
    wr = lay.dense()[0]
    lg = oracle.router_logits_np(x, wr, lay.bias_host)
    ref = oracle.select_topk(lg, lay.d.top_k)
    tol = boundary_tol(lg)
    same = np.all(idx == ref, axis=1)
    amb = topk_gap_ambiguous(lg, lay.d.top_k, tol)
    assert np.all(same | amb), f"{int((~same & ~amb).sum())} tokens select other experts"
    for t in np.nonzero(~same)[0]:
        assert selection_valid(lg[t], idx[t], lay.d.top_k, 2 * tol[t]), t
    assert np.all(np.diff(idx, axis=1) > 0)
    return int((~same).sum())


def check_permutation(d, idx: np.ndarray, ws=None):
    """k3moe_permute of a selection against the oracle's counting sort of the same selection
    (integer work on the same input: bit-exact). Returns the expert offsets."""
    T = idx.shape[0]
    dm = dims(d)
    off = torch.empty(d.n_experts + 1, dtype=torch.int32, device=DEV)
    rt, rs, sr = (torch.empty(T * d.top_k, dtype=torch.int32, device=DEV) for _ in range(3))
    wsb, n = ws if ws is not None else workspace(dm, T)
    idd = up(np.ascontiguousarray(idx, np.int32))
    k3.k3moe_permute(dm, idd.data_ptr(), T, off.data_ptr(), rt.data_ptr(), rs.data_ptr(), sr.data_ptr(),
                     wsb.data_ptr(), n, stream())
    check_ok(wsb)
    want = oracle.permute(idx, d.n_experts)
    for g, r in zip((off, rt, rs, sr), want):
        np.testing.assert_array_equal(g.cpu().numpy(), r)
    return want[0]


def check_rounding_straddles(got_bits: np.ndarray, exact: np.ndarray, mag: np.ndarray, rel: float = 2.0**-20):
    """bf16 results of fp32 sums against the exact sums: every element must be the bf16 rounding
    of some value within rel * mag of the exact sum (mag = the sum of |terms|, which bounds an
    fp32 sum's error), i.e. lie between the roundings of exact - rel * mag and exact + rel * mag.
    Elsewhere than near a rounding midpoint (or near zero) that interval holds one bf16 value,
    the correctly rounded one. Returns the number of elements per row that differ from the
    correctly rounded exact sums."""
    dlt = rel * mag
    g = oracle.bf16_to_f64(got_bits)
    lo = oracle.bf16_to_f64(bf16_from_exact(exact - dlt))
    hi = oracle.bf16_to_f64(bf16_from_exact(exact + dlt))
    bad = ~((lo <= g) & (g <= hi))
    assert not bad.any(), (int(bad.sum()), exact[bad][:4], g[bad][:4])
    return (got_bits != bf16_from_exact(exact)).sum(axis=-1)


def bf16_from_exact(v: np.ndarray) -> np.ndarray:
    return oracle.bf16_from_f64_np(v)
