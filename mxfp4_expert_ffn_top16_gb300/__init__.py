"""Python binding of libk3moe: one Stable-LatentMoE routed-expert layer with MXFP4 experts,
run by hand-written CUDA kernels for sm_103a.

Argument marshalling only. Every function here forwards to the C entry point of the same
name in ``libk3moe.so`` (declared in ``include/k3moe.h``); all device work happens in the
library's kernels. Pointers are plain integers (``tensor.data_ptr()``), streams are
``cudaStream_t`` handles as integers (``torch.cuda.current_stream().cuda_stream``).

If the library has not been built, ``lib()`` raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_LIBDIR = os.path.join(_HERE, "_lib")
LIB_PATH = os.path.join(_LIBDIR, "libk3moe.so")

SOURCES = ["k3moe_api.cu", "k_dense_gemv.cu", "k_expert_gemv.cu", "k_route.cu", "k_misc.cu",
           "k_tma.cu", "k_umma_dense.cu", "k_umma_expert.cu", "k_umma_wm.cu", "k_umma_wn.cu",
           "k3moe_noalloc.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-I" + _INCLUDE]

STATUS = {0: "K3MOE_OK", 1: "K3MOE_E_NULL", 2: "K3MOE_E_SHAPE", 3: "K3MOE_E_ALIGN",
          4: "K3MOE_E_WORKSPACE", 5: "K3MOE_E_MODE", 6: "K3MOE_E_CUDA", 7: "K3MOE_E_TIMEOUT",
          8: "K3MOE_E_DEVICE", 9: "K3MOE_E_SCRATCH", 10: "K3MOE_E_HOSTMEM"}
K3MOE_OK = 0

# Exported symbols (kept in step with include/k3moe.h; a CPU test checks both).
EXPORTS = ["k3moe_workspace_size", "k3moe_route", "k3moe_permute", "k3moe_project",
           "k3moe_expert_ffn_mxfp4", "k3moe_combine", "k3moe_layer_forward", "k3moe_check",
           "k3moe_status_string", "k3moe_profile", "k3moe_profile_name", "k3moe_route_noalloc",
           "k3moe_layer_stats", "k3moe_selftest_timeout", "k3moe_selftest_occupy", "k3moe_layer_saliency",
           "k3moe_layer_init", "k3moe_layer_run", "k3moe_layer_run_host", "k3moe_layer_free"]


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, jobs: int = 8) -> str:
    """Compile the CUDA sources for sm_103a and link libk3moe.so (in-tree)."""
    objdir = os.path.join(_LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    headers = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(_INCLUDE, "k3moe.h"))

    def compile_one(src):
        s = os.path.join(_CSRC, src)
        o = os.path.join(objdir, src.replace(".cu", ".o"))
        if force or not _newer(o, [s] + headers):
            subprocess.check_call(["nvcc", *NVCC_FLAGS, "-c", s, "-o", o])
        return o

    with ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or not _newer(LIB_PATH, objs):
        subprocess.check_call(["nvcc", "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-o", LIB_PATH, *objs])
    return LIB_PATH


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "latent", "inter", "n_experts", "top_k", "act", "actq", "n_shared",
                 "shared_inter")]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "router_bias", "w_in", "w_out", "gate_q", "gate_s", "up_q", "up_s",
                 "down_q", "down_s", "w_shared_gate", "w_shared_up", "w_shared_down")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libk3moe is not built ({LIB_PATH} missing); run "
                               "mxfp4_expert_ffn_top16_gb300.build() on a machine with nvcc")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "k3moe_workspace_size": [p, i32, p],
            "k3moe_route": [p, p, i32, p, p, p, p, p, p, sz, p],
            "k3moe_permute": [p, p, i32, p, p, p, p, p, sz, p],
            "k3moe_project": [p, p, i32, i32, i32, p, p, sz, p],
            "k3moe_expert_ffn_mxfp4": [p, p, p, i32, p, p, p, p, sz, p],
            "k3moe_combine": [p, p, p, p, i32, p, p],
            "k3moe_layer_forward": [p, p, p, i32, p, p, p, p, sz, p],
            "k3moe_check": [p, p],
            "k3moe_route_noalloc": [p, p, i32, p, p, p, p, p, p],
            "k3moe_layer_stats": [p, i32, p, sz, p, p, p],
            "k3moe_selftest_timeout": [p, p],
            "k3moe_selftest_occupy": [i32, i32, p],
            "k3moe_layer_saliency": [p, i32, p, p, p, sz, p, p],
            "k3moe_layer_init": [p, p, p, p],
            "k3moe_layer_run": [p, p, i32, p, p, p, p, sz, p],
            "k3moe_layer_run_host": [p, p, i32, p, p, p, p, sz, p],
            "k3moe_layer_free": [p],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = st
        L.k3moe_status_string.argtypes = [st]
        L.k3moe_status_string.restype = ctypes.c_char_p
        L.k3moe_profile.argtypes = [i32, i32, p, p]
        L.k3moe_profile.restype = st
        L.k3moe_profile_name.argtypes = [i32]
        L.k3moe_profile_name.restype = ctypes.c_char_p
        _lib = L
    return _lib


class K3moeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


def _ck(status: int, where: str, check: bool):
    if check and status != K3MOE_OK:
        raise K3moeError(status, where)
    return status


def status_string(status: int) -> str:
    return lib().k3moe_status_string(status).decode()


def _ref(s):
    return None if s is None else ctypes.byref(s)


# ---------------------------------------------------------------- entry points (same names)
def k3moe_workspace_size(dims: Dims, max_tokens: int) -> int:
    out = ctypes.c_size_t(0)
    _ck(lib().k3moe_workspace_size(_ref(dims), max_tokens, ctypes.byref(out)),
        "k3moe_workspace_size", True)
    return out.value


def k3moe_route(dims, x, T, w_router, bias, logits, topk_idx, topk_w, ws, ws_bytes, stream=0,
                check=True):
    return _ck(lib().k3moe_route(_ref(dims), x, T, w_router, bias, logits, topk_idx, topk_w, ws,
                                 ws_bytes, stream), "k3moe_route", check)


def k3moe_route_noalloc(dims, x, T, w_router, bias, topk_idx, topk_w, err_word=None, stream=0,
                        check=True):
    """k3moe_route without a workspace (logits in the library's fixed scratch)."""
    return _ck(lib().k3moe_route_noalloc(_ref(dims), x, T, w_router, bias, topk_idx, topk_w, err_word,
                                         stream), "k3moe_route_noalloc", check)


def k3moe_permute(dims, topk_idx, T, expert_offsets, row_token, row_slot, slot_row, ws, ws_bytes,
                  stream=0, check=True):
    return _ck(lib().k3moe_permute(_ref(dims), topk_idx, T, expert_offsets, row_token, row_slot,
                                   slot_row, ws, ws_bytes, stream), "k3moe_permute", check)


def k3moe_project(W, x, T, N, K, out, ws, ws_bytes, stream=0, check=True):
    return _ck(lib().k3moe_project(W, x, T, N, K, out, ws, ws_bytes, stream), "k3moe_project", check)


def k3moe_expert_ffn_mxfp4(dims, weights, z, T, expert_offsets, row_token, o_rows, ws, ws_bytes,
                           stream=0, check=True):
    return _ck(lib().k3moe_expert_ffn_mxfp4(_ref(dims), _ref(weights), z, T, expert_offsets,
                                            row_token, o_rows, ws, ws_bytes, stream),
               "k3moe_expert_ffn_mxfp4", check)


def k3moe_combine(dims, o_rows, slot_row, topk_w, T, c, stream=0, check=True):
    return _ck(lib().k3moe_combine(_ref(dims), o_rows, slot_row, topk_w, T, c, stream),
               "k3moe_combine", check)


def k3moe_layer_forward(dims, weights, x, T, y, topk_idx_out, topk_w_out, ws, ws_bytes, stream=0,
                        check=True):
    return _ck(lib().k3moe_layer_forward(_ref(dims), _ref(weights), x, T, y, topk_idx_out,
                                         topk_w_out, ws, ws_bytes, stream),
               "k3moe_layer_forward", check)


def k3moe_layer_init(dims, weights, stream=0):
    """A prepared-layer handle (an integer) for k3moe_layer_run; release it with k3moe_layer_free.
    dims and weights are copied into the handle; the weight buffers must outlive it."""
    h = ctypes.c_void_p()
    _ck(lib().k3moe_layer_init(_ref(dims), _ref(weights), ctypes.byref(h), stream), "k3moe_layer_init", True)
    return h.value


def k3moe_layer_run(layer, x, T, y, topk_idx_out, topk_w_out, ws, ws_bytes, stream=0, check=True):
    return _ck(lib().k3moe_layer_run(layer, x, T, y, topk_idx_out, topk_w_out, ws, ws_bytes, stream),
               "k3moe_layer_run", check)


def k3moe_layer_run_host(layer, x_host, T, y_host, topk_idx_out, topk_w_out, ws, ws_bytes, stream=0, check=True):
    """k3moe_layer_run with x and y in page-locked host memory (e.g. torch pinned tensors)."""
    return _ck(lib().k3moe_layer_run_host(layer, x_host, T, y_host, topk_idx_out, topk_w_out, ws, ws_bytes, stream),
               "k3moe_layer_run_host", check)


def k3moe_layer_free(layer):
    return _ck(lib().k3moe_layer_free(layer), "k3moe_layer_free", True)


def k3moe_layer_stats(dims, T, ws, ws_bytes, stream=0):
    """(distinct experts selected in the last step, the expert bytes that step read)."""
    dd = ctypes.c_int32(0)
    eb = ctypes.c_int64(0)
    _ck(lib().k3moe_layer_stats(_ref(dims), T, ws, ws_bytes, stream, ctypes.byref(dd), ctypes.byref(eb)),
        "k3moe_layer_stats", True)
    return dd.value, eb.value


def k3moe_selftest_timeout(ws, stream=0):
    """Enqueues the failure-path self test (a bounded wait that runs out, about 2 s)."""
    return _ck(lib().k3moe_selftest_timeout(ws, stream), "k3moe_selftest_timeout", True)


def k3moe_layer_saliency(dims, T, topk_idx, topk_w, ws, ws_bytes, saliency, stream=0, check=True):
    """Adds the last layer step's REAP saliency sums (w * ||o||_2 per expert) to saliency [E] fp64."""
    return _ck(lib().k3moe_layer_saliency(_ref(dims), T, topk_idx, topk_w, ws, ws_bytes, saliency, stream),
               "k3moe_layer_saliency", check)


def k3moe_selftest_occupy(n_ctas, ms, stream=0):
    """Enqueues n_ctas CTAs that each hold most of an SM's shared memory for ms milliseconds."""
    return _ck(lib().k3moe_selftest_occupy(n_ctas, ms, stream), "k3moe_selftest_occupy", True)


def k3moe_check(ws, stream=0):
    return lib().k3moe_check(ws, stream)


def k3moe_profile(mode: int, n: int = 32):
    """mode 1: start recording; mode 0: stop and return {kernel name: (total ms, launches)}."""
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    _ck(lib().k3moe_profile(mode, n, ms, cnt), "k3moe_profile", True)
    if mode == 1:
        return None
    out = {}
    for i in range(n):
        name = lib().k3moe_profile_name(i)
        if name is None:
            break
        out[name.decode()] = (float(ms[i]), int(cnt[i]))
    return out
