"""Shared helpers of the GPU tests: device layers filled by the seeded generator, the matching
oracle layer built from host-generated tensors, and comparison rules.

Inputs reach the oracle only from the host generator (synth, host side) and reach the GPU
from the device generator or a host->device copy of the same host arrays; nothing the CUDA
library computes is fed to the oracle.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import mxfp4_expert_ffn_top16_gb300 as k3
import oracle
import synth

DEV = torch.device("cuda:0")
NAMES = oracle.ExpertTables.NAMES

# Tolerances (layer outputs within relative L2 error 2e-3 of the oracle; indices bit-exact).
# REL_L2 bounds the relative L2 error of a whole compared output (all compared tokens).
# Per token the layer's four bf16 rounding points (z, GLU output, combine, y) turn a
# one-fp32-ulp difference upstream into ~1e-3 of rounding noise on that token, so a single
# token is held to the looser PER_TOKEN guard.
REL_L2 = 2e-3
PER_TOKEN = 5e-3
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
        ids = range(self.d.n_experts) if experts is None else experts
        ex = {int(e): self.expert_host(int(e)) for e in ids}
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


def topk_gap_ambiguous(logits: np.ndarray, k: int, tol: np.ndarray | float) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest oracle logits are closer than tol: there the
    selection at the boundary is decided below the precision of fp32 logits."""
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
