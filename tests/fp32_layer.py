"""A plain fp32 evaluation of the routed-expert layer (torch on the CPU), with the layer's bf16
rounding points (z, the GLU output a, the combined c, y) and fp32 everywhere else.

Test infrastructure for the tolerance reading: it is what "the layer with fp32 accumulation"
computes when nothing but the order of fp32 sums differs from the exact statement, so its
distance from the oracle (exact sums, then the same roundings) is the distance that fp32
accumulation alone produces. It shares no code with the CUDA library or with the oracle; its
decode of the MXFP4 experts follows the pages' description directly (nibble 2j is the low
nibble of byte j, value table of the e2m1 format, one e8m0 exponent per 32 along K)."""
from __future__ import annotations

import numpy as np
import torch

# e2m1 values, OCP MX v1.0 (codes 0..15)
_E2M1 = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float32)


def _bf16(t: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16 (round to nearest even) -> fp32."""
    return t.to(torch.bfloat16).to(torch.float32)


def _f32(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy((np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).copy())


def decode(q: np.ndarray, s: np.ndarray) -> torch.Tensor:
    q = torch.from_numpy(np.asarray(q, np.uint8).astype(np.int64))
    N = q.shape[0]
    codes = torch.stack([q & 15, q >> 4], dim=-1).reshape(N, -1)
    scale = torch.pow(2.0, torch.from_numpy(np.asarray(s, np.float32)) - 127.0)
    return (_E2M1[codes].reshape(N, scale.shape[1], 32) * scale[:, :, None]).reshape(N, -1)


def mxfp8(v: torch.Tensor) -> torch.Tensor:
    """MXFP8 round trip along the last axis in blocks of 32 (OCP MX v1.0: shared exponent
    floor(log2 amax) - 8, elements rounded to E4M3 nearest-even, saturating at +-448)."""
    sh = v.shape
    b = v.reshape(-1, 32)
    amax = b.abs().amax(dim=1, keepdim=True)
    X = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, 1.0))) - 8, -127.0)
    X = X.clamp(-127, 127)
    q = (b * torch.pow(2.0, -X)).clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float32)
    return (q * torch.pow(2.0, X)).reshape(sh)


_E2M1_POS = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=torch.float32)


def mxfp4(v: torch.Tensor) -> torch.Tensor:
    """MXFP4 round trip along the last axis in blocks of 32 (OCP MX v1.0: shared exponent
    floor(log2 amax) - 2, elements rounded to the nearest e2m1 value, ties to the even code,
    saturating at +-6)."""
    sh = v.shape
    b = v.reshape(-1, 32)
    amax = b.abs().amax(dim=1, keepdim=True)
    X = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, 1.0))) - 2, -127.0).clamp(-127, 127)
    a = (b.abs() * torch.pow(2.0, -X)).clamp(max=6.0)
    dist = (a[..., None] - _E2M1_POS).abs()
    best = dist.min(dim=-1, keepdim=True).values
    codes = torch.arange(8)
    # among equally near values, the even code
    cand = torch.where(dist == best, codes + 16 * (codes % 2), 99)
    q = _E2M1_POS[(cand.argmin(dim=-1)) % 16]
    return (torch.sign(b) * q * torch.pow(2.0, X)).reshape(sh)


def forward(d, w_router, w_in, w_out, experts: dict, x: np.ndarray, idx: np.ndarray, wts: np.ndarray,
            actq: int = 0) -> np.ndarray:
    """y (bf16 bits) for tokens x with the selection idx [T][k] and routing weights wts [T][k]
    (taken from the oracle so that only the fp32 arithmetic of the rest differs). actq = 1:
    MXFP8 activations, 2: MXFP4 activations (z and the GLU output go through that round trip)."""
    q = mxfp8 if actq == 1 else (mxfp4 if actq == 2 else (lambda t: t))
    X = _f32(x)
    z = q(_bf16(X @ _f32(w_in).T))
    T, k = idx.shape
    o = torch.zeros(T, k, d.latent)
    for e in np.unique(idx):
        t, j = np.nonzero(idx == e)
        ex = experts[int(e)]
        G, U = decode(ex["gate_q"], ex["gate_s"]), decode(ex["up_q"], ex["up_s"])
        D = decode(ex["down_q"], ex["down_s"])
        zz = z[torch.from_numpy(t)]
        g, u = zz @ G.T, zz @ U.T
        a = q(_bf16(g / (1 + torch.exp(-g)) * u))
        o[torch.from_numpy(t), torch.from_numpy(j)] = a @ D.T
    W = torch.from_numpy(np.asarray(wts, np.float32))
    c = _bf16((W[:, :, None] * o).sum(1))
    y = _bf16(c @ _f32(w_out).T)
    return (y.numpy().view(np.uint32) >> 16).astype(np.uint16)
