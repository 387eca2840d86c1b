"""The C ABI without a GPU: the library builds and loads, exports every function that
include/k3moe.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import mxfp4_expert_ffn_top16_gb300 as k3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    k3.build()
    return k3.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function(L):
    declared = header_functions()
    assert declared, "no declarations parsed"
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(k3.EXPORTS) == declared


def test_status_strings(L):
    for code, name in k3.STATUS.items():
        assert k3.status_string(code).startswith(name)


K3 = dict(hidden=7168, latent=3584, inter=3072, n_experts=896, top_k=16, act=0, actq=0)


def dims(**kw):
    v = dict(K3)
    v.update(kw)
    return k3.Dims(**v)


def test_workspace_size_monotone(L):
    a = k3.k3moe_workspace_size(dims(), 1)
    b = k3.k3moe_workspace_size(dims(), 64)
    c = k3.k3moe_workspace_size(dims(), 4096)
    assert 256 < a < b < c


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=7000), 2), (dict(latent=0), 2), (dict(inter=100), 2), (dict(n_experts=2000), 2),
    (dict(top_k=0), 2), (dict(top_k=33), 2), (dict(n_experts=8, top_k=9), 2),
    (dict(act=1), 5), (dict(actq=3), 5), (dict(actq=2, latent=3648), 5), (dict(actq=2, inter=3136), 5),
    (dict(actq=2), 0)])
def test_bad_dims_rejected(L, kw, status):
    out = ctypes.c_size_t(0)
    assert L.k3moe_workspace_size(ctypes.byref(dims(**kw)), 4, ctypes.byref(out)) == status


def test_null_misaligned_and_small_workspace_rejected(L):
    d = dims()
    good = 0x10000
    # null inputs
    assert k3.k3moe_route(d, None, 4, good, None, None, good, good, good, 1 << 30, check=False) == 1
    assert L.k3moe_route(None, good, 4, good, None, None, good, good, good, 1 << 30, None) == 1
    # misaligned
    assert k3.k3moe_route(d, good + 2, 4, good, None, None, good, good, good, 1 << 30, check=False) == 3
    # workspace too small / missing
    assert k3.k3moe_route(d, good, 4, good, None, None, good, good, good, 100, check=False) == 4
    assert k3.k3moe_route(d, good, 4, good, None, None, good, good, None, 1 << 30, check=False) == 4
    # negative T
    assert k3.k3moe_permute(d, good, -1, good, good, good, good, good, 1 << 30, check=False) == 2
    # projection shape rules
    assert k3.k3moe_project(good, good, 1, 100, 64, good, good, 256, check=False) == 2
    w = k3.Weights(good, None, good, good, good, None, good, good, good, good)
    assert k3.k3moe_expert_ffn_mxfp4(d, w, good, 1, good, good, good, good, 1 << 30, check=False) == 1
    w.gate_s = good + 8
    assert k3.k3moe_layer_forward(d, w, good, 1, good, None, None, good, 1 << 30, check=False) == 3
    # SiTU-GLU has no formula on the pages: refused
    assert k3.k3moe_layer_forward(dims(act=1), w, good, 1, good, None, None, good, 1 << 30,
                                  check=False) == 5


def test_shared_expert_dims_and_workspace(L):
    """Shared experts: n_shared in 0..8, n_shared * shared_inter a positive multiple of 64; their
    buffers ([T][S] gate and up fp32, GLU output bf16) grow the workspace by 10 * T * S bytes at
    most (plus alignment)."""
    T = 64
    base = k3.k3moe_workspace_size(dims(), T)
    with_sh = k3.k3moe_workspace_size(dims(n_shared=2, shared_inter=3072), T)
    S = 2 * 3072
    assert 10 * T * S <= with_sh - base <= 10 * T * S + 3 * 256
    out = ctypes.c_size_t(0)
    for kw in (dict(n_shared=9, shared_inter=64), dict(n_shared=-1, shared_inter=64),
               dict(n_shared=2, shared_inter=0), dict(n_shared=3, shared_inter=20)):
        assert L.k3moe_workspace_size(ctypes.byref(dims(**kw)), 4, ctypes.byref(out)) == 2, kw
    assert L.k3moe_workspace_size(ctypes.byref(dims(n_shared=1, shared_inter=64)), 4, ctypes.byref(out)) == 0


def test_shared_expert_weights_checked(L):
    good = 0x10000
    d = dims(n_shared=2, shared_inter=64)
    w = k3.Weights(good, None, good, good, good, good, good, good, good, good)
    # shared pointers missing
    assert k3.k3moe_layer_forward(d, w, good, 1, good, None, None, good, 1 << 30, check=False) == 1
    w.w_shared_gate, w.w_shared_up, w.w_shared_down = good, good + 4, good
    assert k3.k3moe_layer_forward(d, w, good, 1, good, None, None, good, 1 << 30, check=False) == 3


def test_layer_stats_arguments(L):
    good = 0x10000
    out = ctypes.c_int32(0)
    assert L.k3moe_layer_stats(None, 1, good, 1 << 30, None, ctypes.byref(out), None) == 1
    assert L.k3moe_layer_stats(ctypes.byref(dims()), -1, good, 1 << 30, None, ctypes.byref(out), None) == 2
    assert L.k3moe_layer_stats(ctypes.byref(dims()), 1, good, 100, None, ctypes.byref(out), None) == 4
    # T = 0: nothing was selected, no device access
    eb = ctypes.c_int64(7)
    assert L.k3moe_layer_stats(ctypes.byref(dims()), 0, good, 1 << 30, None, ctypes.byref(out),
                               ctypes.byref(eb)) == 0
    assert out.value == 0 and eb.value == 0


def test_selftest_occupy_arguments(L):
    """Out-of-range requests are refused before anything is launched (no GPU needed)."""
    for n, ms in ((0, 10), (5000, 10), (4, 0), (4, 10001)):
        assert L.k3moe_selftest_occupy(n, ms, None) == 2


def test_layer_saliency_arguments(L):
    """Checks before any launch (no GPU needed): dims, the accumulator, alignment, workspace."""
    dm = k3.Dims(7168, 3584, 3072, 896, 16, 0, 0, 0, 0)
    good = 1 << 16
    n = k3.k3moe_workspace_size(dm, 4)
    assert L.k3moe_layer_saliency(ctypes.byref(dm), 4, None, None, good, n, None, None) == 1
    assert L.k3moe_layer_saliency(ctypes.byref(dm), 4, None, None, good, n, good + 8, None) == 3
    assert L.k3moe_layer_saliency(ctypes.byref(dm), 4, None, None, good, n - 1, good, None) == 4
    assert L.k3moe_layer_saliency(ctypes.byref(dm), -1, None, None, good, n, good, None) == 2
    assert L.k3moe_layer_saliency(ctypes.byref(dm), 0, None, None, good, n, good, None) == 0


def test_prepared_layer_arguments(L):
    """k3moe_layer_init / k3moe_layer_run / k3moe_layer_free reject bad arguments before any
    allocation or launch (no GPU needed); freeing NULL is allowed."""
    good = 1 << 16
    h = ctypes.c_void_p(123)
    w = k3.Weights(good, None, good, good, good, good, good, good, good, good)
    assert L.k3moe_layer_init(ctypes.byref(dims()), ctypes.byref(w), None, None) == 1
    assert L.k3moe_layer_init(ctypes.byref(dims(latent=100)), ctypes.byref(w), ctypes.byref(h), None) == 2
    assert h.value is None  # a failed init leaves no handle
    w.up_s = good + 4
    assert L.k3moe_layer_init(ctypes.byref(dims()), ctypes.byref(w), ctypes.byref(h), None) == 3
    w.up_s = None
    assert L.k3moe_layer_init(ctypes.byref(dims()), ctypes.byref(w), ctypes.byref(h), None) == 1
    assert L.k3moe_layer_init(ctypes.byref(dims(act=1)), ctypes.byref(w), ctypes.byref(h), None) == 5
    assert L.k3moe_layer_run(None, good, 1, good, None, None, good, 1 << 30, None) == 1
    assert L.k3moe_layer_run_host(None, good, 1, good, None, None, good, 1 << 30, None) == 1
    assert L.k3moe_layer_free(None) == 0
