"""Python face of the reference oracle (``k3moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline may import this; the library never does. It computes one Stable-LatentMoE
routed-expert layer with MXFP4 experts in plain scalar C with double accumulation.

Every function takes and returns numpy arrays; bf16 values travel as uint16 bit patterns.
Parity status: every step is pinned by the ``-m "not gpu"`` tests except the SiTU-GLU
activation, which the pages name without a formula (parity unpinned; the oracle refuses
act != 0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libk3moe_oracle.so")


def build(force: bool = False) -> str:
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", _LIB, _SRC, "-lm"])
    return _LIB


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "latent", "inter", "n_experts", "top_k", "act", "actq", "n_shared",
                 "shared_inter")]


class Weights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w_in", ctypes.c_void_p), ("w_out", ctypes.c_void_p),
                ("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p),
                ("up_q", ctypes.c_void_p), ("up_s", ctypes.c_void_p),
                ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p),
                ("w_sgate", ctypes.c_void_p), ("w_sup", ctypes.c_void_p), ("w_sdown", ctypes.c_void_p)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.k3o_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.k3o_bf16_to_double.restype = d
        L.k3o_bf16_from_double.argtypes = [d]
        L.k3o_bf16_from_double.restype = ctypes.c_uint16
        for f in ("k3o_e2m1", "k3o_e8m0", "k3o_e4m3"):
            getattr(L, f).argtypes = [i]
            getattr(L, f).restype = d
        L.k3o_e4m3_encode.argtypes = [d]
        L.k3o_e4m3_encode.restype = i
        L.k3o_mxfp8_block.argtypes = [p, p, p]
        L.k3o_mxfp8_roundtrip.argtypes = [p, i]
        L.k3o_e2m1_encode.argtypes = [d]
        L.k3o_e2m1_encode.restype = i
        L.k3o_mxfp4_block.argtypes = [p, p, p]
        L.k3o_mxfp4_roundtrip.argtypes = [p, i]
        L.k3o_mx_weight.argtypes = [p, p, i]
        L.k3o_mx_weight.restype = d
        L.k3o_dequant.argtypes = [p, p, i, i, p]
        L.k3o_dequant_row.argtypes = [p, p, i, p]
        L.k3o_expert_params.argtypes = [p]
        L.k3o_expert_params.restype = ctypes.c_int64
        L.k3o_expert_bytes.argtypes = [p]
        L.k3o_expert_bytes.restype = ctypes.c_int64
        L.k3o_router_logits.argtypes = [p, p, i, p, p, p]
        L.k3o_select_topk.argtypes = [p, i, i, i, p]
        L.k3o_route_weights.argtypes = [p, p, i, i, i, p]
        L.k3o_permute.argtypes = [p, i, i, i, p, p, p, p]
        L.k3o_dense_proj.argtypes = [p, p, i, i, i, p, p]
        L.k3o_expert_row.argtypes = [p, p, i, p, p, p]
        L.k3o_expert_row.restype = i
        L.k3o_combine_token.argtypes = [i, i, p, p, p, p]
        L.k3o_shared_ffn.argtypes = [p, p, p, p, p]
        L.k3o_shared_ffn.restype = i
        L.k3o_layer_forward.argtypes = [p, p, p, i, p, p, p, p, p, p, i]
        L.k3o_layer_forward.restype = i
        L.k3o_max_threads.restype = i
        L.k3o_saliency_accumulate.argtypes = [p, i, p, p, p, p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats
def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_f64(x) -> np.ndarray:
    x = np.asarray(x, np.float64)
    f = lib().k3o_bf16_from_double
    return np.array([f(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)


def e2m1(code: int) -> float:
    return lib().k3o_e2m1(code)


def e8m0(e: int) -> float:
    return lib().k3o_e8m0(e)


def e4m3(code: int) -> float:
    return lib().k3o_e4m3(code)


def e4m3_encode(v: float) -> int:
    return lib().k3o_e4m3_encode(v)


def mxfp8_block(v):
    v = _c(v, np.float64)
    assert v.shape == (32,)
    codes = np.empty(32, np.uint8)
    sc = np.empty(1, np.uint8)
    lib().k3o_mxfp8_block(v.ctypes.data, codes.ctypes.data, sc.ctypes.data)
    return codes, int(sc[0])


def mxfp8_roundtrip(v):
    v = _c(v, np.float64).copy()
    lib().k3o_mxfp8_roundtrip(v.ctypes.data, v.size)
    return v


def e2m1_encode(v: float) -> int:
    return lib().k3o_e2m1_encode(v)


def mxfp4_block(v):
    v = _c(v, np.float64)
    assert v.shape == (32,)
    codes = np.empty(32, np.uint8)
    sc = np.empty(1, np.uint8)
    lib().k3o_mxfp4_block(v.ctypes.data, codes.ctypes.data, sc.ctypes.data)
    return codes, int(sc[0])


def mxfp4_roundtrip(v):
    v = _c(v, np.float64).copy()
    lib().k3o_mxfp4_roundtrip(v.ctypes.data, v.size)
    return v


def dequant(q, s, N, K) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    out = np.empty((N, K), np.float64)
    lib().k3o_dequant(q.ctypes.data, s.ctypes.data, N, K, out.ctypes.data)
    return out


def dequant_row(q_row, s_row, K) -> np.ndarray:
    q_row, s_row = _c(q_row, np.uint8), _c(s_row, np.uint8)
    out = np.empty(K, np.float64)
    lib().k3o_dequant_row(q_row.ctypes.data, s_row.ctypes.data, K, out.ctypes.data)
    return out


def mx_weight(q_row, s_row, j) -> float:
    q_row, s_row = _c(q_row, np.uint8), _c(s_row, np.uint8)
    return lib().k3o_mx_weight(q_row.ctypes.data, s_row.ctypes.data, j)


def make_dims(d, act=0, actq=0, n_shared=0, shared_inter=0) -> Dims:
    return Dims(d.hidden, d.latent, d.inter, d.n_experts, d.top_k, act, actq, n_shared, shared_inter)


def expert_params(d) -> int:
    return lib().k3o_expert_params(ctypes.byref(make_dims(d)))


def expert_bytes(d) -> int:
    return lib().k3o_expert_bytes(ctypes.byref(make_dims(d)))


# ------------------------------------------------------------------ steps
def router_logits(d, x, w_router, bias=None) -> np.ndarray:
    x, wr = _c(x, np.uint16), _c(w_router, np.uint16)
    T = x.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, d.n_experts), np.float64)
    lib().k3o_router_logits(ctypes.byref(make_dims(d)), x.ctypes.data, T, wr.ctypes.data,
                            _ptr(b), out.ctypes.data)
    return out


def router_logits_np(x, w_router, bias=None) -> np.ndarray:
    """Router logits for many tokens: the same sum as router_logits, taken as one float64
    matrix product of the bf16 values (a library matmul as the summation step)."""
    lg = bf16_to_f64(x) @ bf16_to_f64(w_router).T
    if bias is not None:
        lg = lg + np.asarray(bias, np.float32).astype(np.float64)
    return lg


def select_topk(logits, k) -> np.ndarray:
    lg = _c(logits, np.float64)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    lib().k3o_select_topk(lg.ctypes.data, T, E, k, idx.ctypes.data)
    return idx


def route_weights(logits, idx) -> np.ndarray:
    lg, idx = _c(logits, np.float64), _c(idx, np.int32)
    T, E = lg.shape
    k = idx.shape[1]
    w = np.empty((T, k), np.float64)
    lib().k3o_route_weights(lg.ctypes.data, idx.ctypes.data, T, E, k, w.ctypes.data)
    return w


def permute(idx, E):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    off = np.empty(E + 1, np.int32)
    rt = np.empty(T * k, np.int32)
    rs = np.empty(T * k, np.int32)
    sr = np.empty(T * k, np.int32)
    lib().k3o_permute(idx.ctypes.data, T, E, k, off.ctypes.data, rt.ctypes.data, rs.ctypes.data,
                      sr.ctypes.data)
    return off, rt, rs, sr


def dense_proj(W, x):
    """out = W x for every token row; returns (double [T][N], bf16 bits [T][N])."""
    W, x = _c(W, np.uint16), _c(x, np.uint16)
    N, K = W.shape
    T = x.shape[0]
    out = np.empty((T, N), np.float64)
    ob = np.empty((T, N), np.uint16)
    lib().k3o_dense_proj(W.ctypes.data, x.ctypes.data, T, N, K, out.ctypes.data, ob.ctypes.data)
    return out, ob


class ExpertTables:
    """Keeps per-expert pointer tables (and the arrays behind them) alive."""

    NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")

    def __init__(self, n_experts: int, experts: dict):
        self.keep = []
        self.tables = {}
        for name in self.NAMES:
            tab = (ctypes.c_void_p * n_experts)()
            for e, t in experts.items():
                a = _c(t[name], np.uint8)
                self.keep.append(a)
                tab[e] = a.ctypes.data
            self.tables[name] = tab

    def fill(self, w: Weights):
        for name in self.NAMES:
            setattr(w, name, ctypes.cast(self.tables[name], ctypes.c_void_p))


class Layer:
    """A layer for the oracle: dense weights (bf16 bits) plus the experts that may be
    selected ({e: {gate_q, gate_s, up_q, up_s, down_q, down_s}})."""

    def __init__(self, d, w_router, w_in, w_out, experts: dict, bias=None, act=0, actq=0, shared=None):
        """shared: None, or (w_sgate [S][H], w_sup [S][H], w_sdown [H][S], n_shared) bf16 bits,
        the n_shared experts stacked along S."""
        self.d = d
        ns, si = 0, 0
        if shared is not None:
            ns = shared[3]
            si = shared[0].shape[0] // ns
        self.dims = make_dims(d, act, actq, ns, si)
        self.wr = _c(w_router, np.uint16)
        self.wi = _c(w_in, np.uint16)
        self.wo = _c(w_out, np.uint16)
        self.bias = None if bias is None else _c(bias, np.float32)
        self.experts = experts
        self.et = ExpertTables(d.n_experts, experts)
        self.w = Weights()
        self.w.w_router = self.wr.ctypes.data
        self.w.router_bias = _ptr(self.bias)
        self.w.w_in = self.wi.ctypes.data
        self.w.w_out = self.wo.ctypes.data
        self.et.fill(self.w)
        self.shared = None
        if shared is not None:
            self.shared = [_c(a, np.uint16) for a in shared[:3]]
            self.w.w_sgate, self.w.w_sup, self.w.w_sdown = (a.ctypes.data for a in self.shared)

    def shared_ffn(self, x_row):
        """The shared experts on one token: (s double [H], stacked GLU outputs bf16 [S])."""
        x = _c(x_row, np.uint16)
        s = np.empty(self.d.hidden, np.float64)
        a = np.empty(max(1, self.dims.n_shared * self.dims.shared_inter), np.uint16)
        if lib().k3o_shared_ffn(ctypes.byref(self.dims), ctypes.byref(self.w), x.ctypes.data,
                                s.ctypes.data, a.ctypes.data) != 0:
            raise ValueError("oracle: unsupported activation")
        return s, a

    def expert_row(self, e, z_row):
        z = _c(z_row, np.uint16)
        o = np.empty(self.d.latent, np.float64)
        a = np.empty(self.d.inter, np.uint16)
        rc = lib().k3o_expert_row(ctypes.byref(self.dims), ctypes.byref(self.w), e, z.ctypes.data,
                                  o.ctypes.data, a.ctypes.data)
        if rc != 0:
            raise ValueError("oracle: unsupported activation")
        return o, a

    def forward(self, x, nthreads=1):
        x = _c(x, np.uint16)
        T = x.shape[0]
        d = self.d
        y = np.empty((T, d.hidden), np.uint16)
        idx = np.empty((T, d.top_k), np.int32)
        wt = np.empty((T, d.top_k), np.float64)
        lg = np.empty((T, d.n_experts), np.float64)
        z = np.empty((T, d.latent), np.uint16)
        c = np.empty((T, d.latent), np.uint16)
        rc = lib().k3o_layer_forward(ctypes.byref(self.dims), ctypes.byref(self.w), x.ctypes.data,
                                     T, y.ctypes.data, idx.ctypes.data, wt.ctypes.data,
                                     lg.ctypes.data, z.ctypes.data, c.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError("oracle: unsupported mode or missing expert tensors")
        return {"y": y, "idx": idx, "w": wt, "logits": lg, "z": z, "c": c}


def combine(o_rows, slot_row, w, T, k):
    """c[t] = bf16(sum_j w[t][j] * o_rows[slot_row[t*k+j]]), j ascending."""
    o_rows = _c(o_rows, np.float64)
    w = _c(w, np.float64)
    L = o_rows.shape[1]
    c = np.empty((T, L), np.uint16)
    for t in range(T):
        rows = [o_rows[slot_row[t * k + j]] for j in range(k)]
        tab = (ctypes.c_void_p * k)(*[r.ctypes.data for r in rows])
        wt = _c(w[t], np.float64)
        ct = np.empty(L, np.uint16)
        lib().k3o_combine_token(L, k, ctypes.cast(tab, ctypes.c_void_p), wt.ctypes.data,
                                ct.ctypes.data, None)
        c[t] = ct
    return c


def max_threads() -> int:
    return lib().k3o_max_threads()


# ------------------------------------------------------------------ batched statement
# The same layer, step for step and with the same rounding points, for checks over thousands of
# tokens: the sums are numpy float64 matrix products (a library routine as the summation step)
# instead of the scalar double loops above, and the experts are decoded once per expert instead
# of once per row. It follows the same passages as k3moe_oracle.c ("kimi-k3-mlx", Architecture
# table and Quantisation tiers; "kimi-k3-in-c", MXFP4 experts). Pinned against the scalar C
# statement (tests/test_oracle_batched_pins.py): same selections, same bf16 values.

_E2M1 = None


def _e2m1_table() -> np.ndarray:
    global _E2M1
    if _E2M1 is None:
        _E2M1 = np.array([e2m1(c) for c in range(16)], np.float64)
    return _E2M1


def bf16_from_f64_np(x) -> np.ndarray:
    """double -> bf16 bits, round to nearest, ties to even, in one step: the rule of
    k3o_bf16_from_double, on whole arrays (8 significant bits; below 2^-126 the fixed quantum
    2^-133; overflow to infinity; NaN -> 0x7fc0)."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(a)                     # a in [2^(e-1), 2^e)
        q = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
        r = np.rint(a / q) * q                 # a / q is exact; rint rounds ties to even
        r = np.where(r >= 2.0**128, np.inf, r)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = bits | np.where(np.signbit(x), np.uint16(0x8000), np.uint16(0))
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)


def dequant_np(q, s) -> np.ndarray:
    """MXFP4 matrix [N][K] to doubles: weight j of a row is the nibble j (low nibble first)
    looked up in the 16-entry e2m1 table, times 2^(s[j/32] - 127) (NaN for s = 255)."""
    q = np.asarray(q, np.uint8)
    s = np.asarray(s, np.uint8)
    N, KB = q.shape
    tab = _e2m1_table()
    pairs = np.stack([tab[np.arange(256) & 0xF], tab[np.arange(256) >> 4]], axis=1)  # byte -> (even, odd)
    sc = np.ldexp(1.0, s.astype(np.int64) - 127)
    sc = np.where(s == 255, np.nan, sc)
    w = pairs[q].reshape(N, KB // 16, 32)
    w *= sc[:, :, None]
    return w.reshape(N, 2 * KB)


def _roundtrip_rows(v: np.ndarray, actq: int) -> np.ndarray:
    """MXFP8 (actq 1) or MXFP4 (actq 2) round trip of every row (blocks of 32 along the row)."""
    if actq == 0:
        return v
    out = np.ascontiguousarray(v, np.float64).copy()
    f = lib().k3o_mxfp8_roundtrip if actq == 1 else lib().k3o_mxfp4_roundtrip
    f(out.ctypes.data, out.size)
    return out


def expert_rows(d, ex, z_bits, actq=0) -> np.ndarray:
    """One expert (tensors ex, as the C statement takes them) on z rows (bf16 bits [n][L]):
    o rows [n][L] (double). Same steps as k3o_expert_row: (MXFP8 / MXFP4 round trip of z),
    g, u = G z, U z; a = bf16(silu(g) * u) (round trip of a); o = D a."""
    L, I = d.latent, d.inter
    zq = _roundtrip_rows(bf16_to_f64(z_bits), actq)
    G = dequant(ex["gate_q"], ex["gate_s"], I, L)
    g = zq @ G.T
    G = dequant(ex["up_q"], ex["up_s"], I, L)
    u = zq @ G.T
    del G
    with np.errstate(over="ignore"):  # exp(-g) = inf for very negative g: silu = -0, as in C
        a = bf16_to_f64(bf16_from_f64_np(g / (1.0 + np.exp(-g)) * u))
    a = _roundtrip_rows(a, actq)
    return a @ dequant(ex["down_q"], ex["down_s"], L, I).T


def _layer_np_tail(layer, xf, z, idx, w, nthreads, rows_fn=None):
    """Given the step's tokens xf (double), z (bf16 bits), a selection idx and its weights w:
    expert rows, combine and latent out. Returns (y bits, c bits, o double [T][k][L]).
    rows_fn(e, z_rows) -> o rows replaces expert_rows (e.g. to run the experts elsewhere)."""
    from concurrent.futures import ThreadPoolExecutor
    d = layer.d
    T, k = idx.shape
    actq = layer.dims.actq
    if rows_fn is None:
        rows_fn = lambda e, zr: expert_rows(d, layer.experts[e], zr, actq)
    o = np.zeros((T, k, d.latent), np.float64)

    def run(e):
        t, j = np.nonzero(idx == e)
        o[t, j] = rows_fn(int(e), z[t])

    with ThreadPoolExecutor(max(1, nthreads)) as pool:
        list(pool.map(run, np.unique(idx)))
    acc = np.zeros((T, d.latent), np.float64)
    for j in range(k):  # slot order, as the scalar combine
        acc += w[:, j:j + 1] * o[:, j]
    c = bf16_from_f64_np(acc)
    yd = bf16_to_f64(c) @ bf16_to_f64(layer.wo).T
    if layer.shared is not None:
        ns, si = layer.dims.n_shared, layer.dims.shared_inter
        sg, su, sd = (bf16_to_f64(a) for a in layer.shared)
        g, u = xf @ sg.T, xf @ su.T
        with np.errstate(over="ignore"):
            a = bf16_to_f64(bf16_from_f64_np(g / (1.0 + np.exp(-g)) * u))
        for j in range(ns):  # each shared expert summed on its own, in expert order
            yd += a[:, j * si:(j + 1) * si] @ sd[:, j * si:(j + 1) * si].T
    return bf16_from_f64_np(yd), c, o


def _layer_forward_np(layer, x, nthreads=8, idx=None, rows_fn=None):
    """Layer.forward for many tokens (see Layer.forward_np)."""
    if layer.dims.act != 0:
        raise ValueError("oracle: unsupported activation")
    d = layer.d
    x = _c(x, np.uint16)
    xf = bf16_to_f64(x)
    lg = xf @ bf16_to_f64(layer.wr).T
    if layer.bias is not None:
        lg = lg + layer.bias.astype(np.float64)
    sel = select_topk(lg, d.top_k) if idx is None else _c(idx, np.int32)
    w = route_weights(lg, sel)
    z = bf16_from_f64_np(xf @ bf16_to_f64(layer.wi).T)
    y, c, o = _layer_np_tail(layer, xf, z, sel, w, nthreads, rows_fn)
    return {"y": y, "idx": sel, "w": w, "logits": lg, "z": z, "c": c, "o": o}


def _forward_np(self, x, nthreads=8, rows_fn=None):
    """The whole layer for many tokens (batched statement): same outputs as forward().
    rows_fn(e, z_rows) -> o rows: optional replacement of expert_rows for expert e."""
    return _layer_forward_np(self, x, nthreads, rows_fn=rows_fn)


def _forward_with_selection(self, x, idx, nthreads=8, rows_fn=None):
    """The layer completed with a given expert selection idx [T][k] (ascending per token)
    instead of its own top-k: weights from the oracle's logits at those experts, then every
    later step as in forward(). For tokens whose k-th and (k+1)-th logits are too close for an
    fp32 computation to order, checked elsewhere to be a valid selection."""
    return _layer_forward_np(self, x, nthreads, idx=idx, rows_fn=rows_fn)


Layer.forward_np = _forward_np
Layer.forward_with_selection = _forward_with_selection


# ------------------------------------------------------------------ REAP saliency
def saliency_accumulate(d, idx, w, o, S=None) -> np.ndarray:
    """k3o_saliency_accumulate: S[e] += w[t][j] * ||o[t][j]||_2 over every (t, j) with
    idx[t][j] = e ("kimi-k3-mlx" digest, REAP pruning: S_j = (1/|C|) sum_x g_j(x) ||e_j(x)||_2;
    the caller divides by |C|). idx [T][k], w [T][k] double, o [T][k][L] double."""
    idx, w, o = _c(idx, np.int32), _c(w, np.float64), _c(o, np.float64)
    T = idx.shape[0]
    S = np.zeros(d.n_experts, np.float64) if S is None else S
    assert S.dtype == np.float64 and S.flags.c_contiguous
    lib().k3o_saliency_accumulate(ctypes.byref(make_dims(d)), T, idx.ctypes.data, w.ctypes.data, o.ctypes.data,
                                  S.ctypes.data)
    return S


def saliency(layer, x, nthreads=8, rows_fn=None) -> np.ndarray:
    """REAP saliency of every expert over the tokens x taken as the calibration set C:
    S_j = (1/|C|) sum_x g_j(x) ||e_j(x)||_2, from the layer's own selection, weights and
    expert outputs."""
    ref = layer.forward_np(x, nthreads=nthreads, rows_fn=rows_fn)
    return saliency_accumulate(layer.d, ref["idx"], ref["w"], ref["o"]) / x.shape[0]
