"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the layer. It defines, for each workload, which
SplitMix64 stream and which value rule fill each tensor (see ``synth_host.c`` for the
rules), and gives two byte-identical implementations: ``host_*`` (C, for the oracle and
for small cases) and ``dev_*`` (CUDA, for the K3-sized expert stores).

Workloads follow the layer the pages describe: Kimi K3's Stable LatentMoE, 896 routed
experts with top-16 selection, a 7168-wide residual and a 3584-wide latent space
(kimi-k3-mlx digest, "Architecture" table; kimi-k3-in-c, "MXFP4" section), with MXFP4
experts of 17,547,264 bytes, i.e. gate/up [3072 x 3584] and down [3584 x 3072].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_HOST_SRC = os.path.join(_HERE, "synth_host.c")
_DEV_SRC = os.path.join(_HERE, "synth_dev.cu")
_HOST_LIB = os.path.join(_LIBDIR, "libk3synth_host.so")
_DEV_LIB = os.path.join(_LIBDIR, "libk3synth_dev.so")

# Stream ids: one independent SplitMix64 stream per tensor.
S_X, S_W_ROUTER, S_W_IN, S_W_OUT = 1, 2, 3, 4
S_GATE_Q, S_GATE_S, S_UP_Q, S_UP_S, S_DOWN_Q, S_DOWN_S = 5, 6, 7, 8, 9, 10
S_BIAS, S_PERM, S_IDX = 11, 12, 13
S_SGATE, S_SUP, S_SDOWN = 14, 15, 16

SIGMA_X = 1.0       # tokens ~N(0, 1)
SIGMA_W = 0.02      # router and latent projections ~N(0, 0.02)
E8M0_LO, E8M0_HI = 120, 127  # expert scales U{120..127}


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def build_host(force: bool = False) -> str:
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or _stale(_HOST_LIB, _HOST_SRC):
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", _HOST_LIB, _HOST_SRC])
    return _HOST_LIB


def build_dev(force: bool = False) -> str:
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or _stale(_DEV_LIB, _DEV_SRC):
        subprocess.check_call(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC",
                               "-gencode", "arch=compute_103a,code=sm_103a",
                               "-o", _DEV_LIB, _DEV_SRC])
    return _DEV_LIB


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        u64, sz, p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        lib.k3s_key.argtypes = [u64, u64]
        lib.k3s_key.restype = u64
        lib.k3s_rand64.argtypes = [u64, u64, u64]
        lib.k3s_rand64.restype = u64
        lib.k3s_fill_bytes.argtypes = [u64, u64, u64, sz, p]
        lib.k3s_fill_uniform_u8.argtypes = [u64, u64, u64, sz, ctypes.c_int, ctypes.c_int, p]
        lib.k3s_fill_uniform_i32.argtypes = [u64, u64, u64, sz, ctypes.c_int64, ctypes.c_int64, p]
        lib.k3s_fill_bf16_normal.argtypes = [u64, u64, u64, sz, ctypes.c_float, p]
        lib.k3s_fill_f32_normal.argtypes = [u64, u64, u64, sz, ctypes.c_float, p]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_dev())
        u64, sz, p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        lib.k3s_dev_fill_bytes.argtypes = [u64, u64, u64, sz, p, p]
        lib.k3s_dev_fill_uniform_u8.argtypes = [u64, u64, u64, sz, ctypes.c_int, ctypes.c_int, p, p]
        lib.k3s_dev_fill_bf16_normal.argtypes = [u64, u64, u64, sz, ctypes.c_float, p, p]
        for f in (lib.k3s_dev_fill_bytes, lib.k3s_dev_fill_uniform_u8, lib.k3s_dev_fill_bf16_normal):
            f.restype = ctypes.c_int
        _dev = lib
    return _dev


# ---------------------------------------------------------------- host fills
def rand64(seed: int, stream: int, n: int) -> int:
    return int(_host_lib().k3s_rand64(seed, stream, n))


def host_bytes(seed, stream, offset, n) -> np.ndarray:
    out = np.empty(n, np.uint8)
    _host_lib().k3s_fill_bytes(seed, stream, offset, n, out.ctypes.data)
    return out


def host_uniform_u8(seed, stream, offset, n, lo, hi) -> np.ndarray:
    out = np.empty(n, np.uint8)
    _host_lib().k3s_fill_uniform_u8(seed, stream, offset, n, lo, hi, out.ctypes.data)
    return out


def host_uniform_i32(seed, stream, offset, n, lo, hi) -> np.ndarray:
    out = np.empty(n, np.int32)
    _host_lib().k3s_fill_uniform_i32(seed, stream, offset, n, lo, hi, out.ctypes.data)
    return out


def host_bf16_normal(seed, stream, offset, n, sigma) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _host_lib().k3s_fill_bf16_normal(seed, stream, offset, n, sigma, out.ctypes.data)
    return out


def host_f32_normal(seed, stream, offset, n, sigma) -> np.ndarray:
    out = np.empty(n, np.float32)
    _host_lib().k3s_fill_f32_normal(seed, stream, offset, n, sigma, out.ctypes.data)
    return out


# ---------------------------------------------------------------- device fills
def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def dev_bytes(seed, stream, offset, n, ptr, cuda_stream=0):
    _check(_dev_lib().k3s_dev_fill_bytes(seed, stream, offset, n, ptr, cuda_stream), "fill_bytes")


def dev_uniform_u8(seed, stream, offset, n, lo, hi, ptr, cuda_stream=0):
    _check(_dev_lib().k3s_dev_fill_uniform_u8(seed, stream, offset, n, lo, hi, ptr, cuda_stream),
           "fill_uniform_u8")


def dev_bf16_normal(seed, stream, offset, n, sigma, ptr, cuda_stream=0):
    _check(_dev_lib().k3s_dev_fill_bf16_normal(seed, stream, offset, n, sigma, ptr, cuda_stream),
           "fill_bf16_normal")


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Dims:
    hidden: int
    latent: int
    inter: int
    n_experts: int
    top_k: int

    # Per-expert tensor sizes in bytes (MXFP4: two codes per byte, one e8m0 per 32 along K).
    @property
    def gate_q_bytes(self):
        return self.inter * self.latent // 2

    @property
    def gate_s_bytes(self):
        return self.inter * self.latent // 32

    @property
    def down_q_bytes(self):
        return self.latent * self.inter // 2

    @property
    def down_s_bytes(self):
        return self.latent * self.inter // 32

    @property
    def expert_bytes(self):
        return 2 * (self.gate_q_bytes + self.gate_s_bytes) + self.down_q_bytes + self.down_s_bytes


TINY = Dims(hidden=256, latent=128, inter=128, n_experts=32, top_k=4)
K3 = Dims(hidden=7168, latent=3584, inter=3072, n_experts=896, top_k=16)


@dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    tokens: int          # tokens per step
    bias: str            # "none" | "normal" | "zipf"
    layers: int = 1
    x_rows: int = 0      # distinct token rows generated (0: = tokens)
    seed: int = 0
    notes: str = ""

    @property
    def x_count(self):
        return self.x_rows or self.tokens


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 8, "none",
                     notes="hidden 256, latent 128, inter 128, 32 experts, top-4, 8 tokens"),
    "decode_b1": Workload("decode_b1", K3, 1, "none", x_rows=1000,
                          notes="K3 layer, 1 token per step, 1000 fresh tokens"),
    "decode_b64": Workload("decode_b64", K3, 64, "normal",
                           notes="K3 layer, 64 tokens per step, per-expert bias ~N(0,1)"),
    "prefill_4k": Workload("prefill_4k", K3, 4096, "zipf",
                           notes="K3 layer, 4096 tokens, Zipf(1.1) log-bias over a permutation"),
    "prefill_32k": Workload("prefill_32k", K3, 32768, "zipf", layers=4,
                            notes="K3 layers x4 (seeds 0..3), 32768 tokens, Zipf and uniform runs"),
    "prefill_32k_uniform": Workload("prefill_32k_uniform", K3, 32768, "none", layers=4,
                                    notes="K3 layers x4, 32768 tokens, unbiased routing"),
}


def zipf_bias(n_experts: int, seed: int, s: float = 1.1) -> np.ndarray:
    """Zipf(s) log-bias: b_e = -s * ln(rank_e), ranks 1..E from a seeded Fisher-Yates
    permutation. Added to the router logits, it makes selection probabilities fall off as
    rank^-s, i.e. Zipf-skewed expert popularity."""
    perm = list(range(n_experts))
    for i in range(n_experts - 1, 0, -1):
        j = (rand64(seed, S_PERM, i) >> 32) * (i + 1) >> 32
        perm[i], perm[j] = perm[j], perm[i]
    rank = np.empty(n_experts, np.float64)
    for pos, e in enumerate(perm):
        rank[e] = pos + 1
    return (-s * np.log(rank)).astype(np.float32)


def router_bias(w: Workload, layer: int = 0):
    seed = w.seed + layer
    if w.bias == "none":
        return None
    if w.bias == "normal":
        return host_f32_normal(seed, S_BIAS, 0, w.dims.n_experts, 1.0)
    if w.bias == "zipf":
        return zipf_bias(w.dims.n_experts, seed)
    raise ValueError(w.bias)


def host_x(w: Workload, first: int = 0, count: int | None = None) -> np.ndarray:
    """Token rows [count][hidden] bf16 bits; x is shared by every layer of a workload."""
    count = w.x_count - first if count is None else count
    h = w.dims.hidden
    return host_bf16_normal(w.seed, S_X, first * h, count * h, SIGMA_X).reshape(count, h)


def host_dense(d: Dims, seed: int):
    """Router [E][H], latent-in [L][H], latent-out [H][L] as bf16 bits."""
    wr = host_bf16_normal(seed, S_W_ROUTER, 0, d.n_experts * d.hidden, SIGMA_W)
    wi = host_bf16_normal(seed, S_W_IN, 0, d.latent * d.hidden, SIGMA_W)
    wo = host_bf16_normal(seed, S_W_OUT, 0, d.hidden * d.latent, SIGMA_W)
    return (wr.reshape(d.n_experts, d.hidden), wi.reshape(d.latent, d.hidden),
            wo.reshape(d.hidden, d.latent))


def host_expert(d: Dims, seed: int, e: int) -> dict:
    """One expert's MXFP4 tensors, row-major with K contiguous:
    gate/up codes [I][L/2], scales [I][L/32]; down codes [L][I/2], scales [L][I/32]."""
    gq, gs, dq, ds = d.gate_q_bytes, d.gate_s_bytes, d.down_q_bytes, d.down_s_bytes
    I, L = d.inter, d.latent
    e = int(e)  # a numpy int32 index would overflow in the byte offsets below
    return {
        "gate_q": host_bytes(seed, S_GATE_Q, e * gq, gq).reshape(I, L // 2),
        "gate_s": host_uniform_u8(seed, S_GATE_S, e * gs, gs, E8M0_LO, E8M0_HI).reshape(I, L // 32),
        "up_q": host_bytes(seed, S_UP_Q, e * gq, gq).reshape(I, L // 2),
        "up_s": host_uniform_u8(seed, S_UP_S, e * gs, gs, E8M0_LO, E8M0_HI).reshape(I, L // 32),
        "down_q": host_bytes(seed, S_DOWN_Q, e * dq, dq).reshape(L, I // 2),
        "down_s": host_uniform_u8(seed, S_DOWN_S, e * ds, ds, E8M0_LO, E8M0_HI).reshape(L, I // 32),
    }


def dev_fill_layer(d: Dims, seed: int, ptrs: dict, cuda_stream=0):
    """Fill a whole layer on the device. ``ptrs`` maps w_router, w_in, w_out, gate_q, gate_s,
    up_q, up_s, down_q, down_s to device addresses of the full [E][...] tensors."""
    E = d.n_experts
    dev_bf16_normal(seed, S_W_ROUTER, 0, E * d.hidden, SIGMA_W, ptrs["w_router"], cuda_stream)
    dev_bf16_normal(seed, S_W_IN, 0, d.latent * d.hidden, SIGMA_W, ptrs["w_in"], cuda_stream)
    dev_bf16_normal(seed, S_W_OUT, 0, d.hidden * d.latent, SIGMA_W, ptrs["w_out"], cuda_stream)
    dev_bytes(seed, S_GATE_Q, 0, E * d.gate_q_bytes, ptrs["gate_q"], cuda_stream)
    dev_bytes(seed, S_UP_Q, 0, E * d.gate_q_bytes, ptrs["up_q"], cuda_stream)
    dev_bytes(seed, S_DOWN_Q, 0, E * d.down_q_bytes, ptrs["down_q"], cuda_stream)
    dev_uniform_u8(seed, S_GATE_S, 0, E * d.gate_s_bytes, E8M0_LO, E8M0_HI, ptrs["gate_s"], cuda_stream)
    dev_uniform_u8(seed, S_UP_S, 0, E * d.gate_s_bytes, E8M0_LO, E8M0_HI, ptrs["up_s"], cuda_stream)
    dev_uniform_u8(seed, S_DOWN_S, 0, E * d.down_s_bytes, E8M0_LO, E8M0_HI, ptrs["down_s"], cuda_stream)


def host_shared(d: Dims, n_shared: int, shared_inter: int, seed: int):
    """Shared experts stacked along S = n_shared * shared_inter, bf16 bits: gate [S][H],
    up [S][H], down [H][S]."""
    S, H = n_shared * shared_inter, d.hidden
    g = host_bf16_normal(seed, S_SGATE, 0, S * H, SIGMA_W).reshape(S, H)
    u = host_bf16_normal(seed, S_SUP, 0, S * H, SIGMA_W).reshape(S, H)
    dn = host_bf16_normal(seed, S_SDOWN, 0, H * S, SIGMA_W).reshape(H, S)
    return g, u, dn


def dev_fill_shared(d: Dims, n_shared: int, shared_inter: int, seed: int, ptrs: dict, cuda_stream=0):
    """Device copy of host_shared: ``ptrs`` maps w_sgate, w_sup, w_sdown to device addresses."""
    S, H = n_shared * shared_inter, d.hidden
    dev_bf16_normal(seed, S_SGATE, 0, S * H, SIGMA_W, ptrs["w_sgate"], cuda_stream)
    dev_bf16_normal(seed, S_SUP, 0, S * H, SIGMA_W, ptrs["w_sup"], cuda_stream)
    dev_bf16_normal(seed, S_SDOWN, 0, H * S, SIGMA_W, ptrs["w_sdown"], cuda_stream)


def dev_fill_x(w: Workload, ptr, first: int = 0, count: int | None = None, cuda_stream=0):
    count = w.x_count - first if count is None else count
    h = w.dims.hidden
    dev_bf16_normal(w.seed, S_X, first * h, count * h, SIGMA_X, ptr, cuda_stream)


def host_topk_sets(seed: int, T: int, E: int, k: int, skew: str = "uniform") -> np.ndarray:
    """Synthetic routing decisions [T][k] int32, k distinct experts per token in ascending
    order, for exercising the permutation on its own. ``skew``: "uniform", "zipf" (popular
    experts by rank^-1.1) or "one" (expert 0 in every token)."""
    out = np.empty((T, k), np.int32)
    if skew == "zipf":
        w = np.arange(1, E + 1, dtype=np.float64) ** -1.1
        cdf = np.cumsum(w) / w.sum()
    ctr = 0
    for t in range(T):
        chosen = set([0]) if skew == "one" else set()
        while len(chosen) < k:
            r = rand64(seed, S_IDX, ctr)
            ctr += 1
            if skew == "zipf":
                u = (r >> 11) * (1.0 / 9007199254740992.0)
                e = int(np.searchsorted(cdf, u, side="right"))
                e = min(e, E - 1)
            else:
                e = (r >> 32) * E >> 32
            chosen.add(int(e))
        out[t] = sorted(chosen)
    return out


def nbytes_layer(d: Dims) -> int:
    return d.n_experts * d.expert_bytes + 2 * (d.n_experts * d.hidden + 2 * d.latent * d.hidden)


def expert_param_count(d: Dims) -> int:
    return 3 * d.latent * d.inter


