"""Parity at the sizes the benchmark runs (slow: minutes of oracle time on the host cores).

prefill 4K: 4096 tokens with the Zipf(1.1) log-bias; every token's selection and the
permutation bit-exact (boundary ties checked for validity), and every token's output against
the oracle, with bf16, MXFP8 and MXFP4 activations.
prefill 32K: four layers with independent weights (seeds 0..3), 32768 tokens each; every
token's selection and the permutation of every layer, and per layer the output of a stratified
1024-token subset: every token of the hottest expert's last chunk of rows, every token of the
coldest selected expert, the first and last tokens, the rest evenly spaced. Tokens are
independent, so the subset check is exact for the tokens it covers.
("kimi-k3-in-c": the single-pass prompt cap of 32,768 tokens.)"""
import os

import numpy as np
import pytest
import torch

import synth
from k3help import (DEV, DeviceLayer, dims, workspace, run_layer, compare_layer, check_selection,
                    check_permutation)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
NCPU = os.cpu_count() or 8
CHUNK = 112  # sorted rows per item of the many-token expert kernel


def _subset(idx: np.ndarray, offsets: np.ndarray, n: int, E: int) -> np.ndarray:
    T, k = idx.shape
    counts = np.diff(offsets)
    hot = int(np.argmax(counts))
    used = np.nonzero(counts)[0]
    cold = int(used[np.argmin(counts[used])])
    r_hot = [r for r in range(offsets[hot], offsets[hot + 1])]
    last = r_hot[(len(r_hot) - 1) // CHUNK * CHUNK:]  # the hottest expert's last chunk of rows
    tok_of_rows = np.nonzero(np.isin(idx, [hot]).any(axis=1))[0]  # tokens of the hot expert, in order
    pick = set(tok_of_rows[[r - offsets[hot] for r in last]].tolist())
    pick |= set(np.nonzero((idx == cold).any(axis=1))[0].tolist())
    pick |= {0, T - 1}
    rest = n - len(pick)
    if rest > 0:
        pick |= set(np.linspace(0, T - 1, rest + 2).astype(int).tolist())
    return np.array(sorted(pick))[: max(n, len(pick))]


def test_prefill_4k_every_token_all_activation_modes():
    w = synth.WORKLOADS["prefill_4k"]
    d = w.dims
    lay = DeviceLayer(d, seed=0, bias=synth.router_bias(w))
    try:
        x = synth.host_x(w)
        T = x.shape[0]
        ws = workspace(dims(d, 0), T)
        for actq in (0, 1, 2):
            lay.actq = actq
            y, idx, _ = run_layer(lay, x, dm=dims(d, actq), ws=ws)
            flips = check_selection(lay, x, idx)
            check_permutation(d, idx, ws=ws)
            err, _ = compare_layer(lay, x, y, idx, np.arange(T), nthreads=NCPU,
                                   what=f"prefill_4k actq={actq}")
            print(f"prefill_4k actq={actq}: {flips} boundary-tie tokens of {T}")
    finally:
        del lay
        torch.cuda.empty_cache()


def test_prefill_32k_four_layers():
    w = synth.WORKLOADS["prefill_32k"]
    d = w.dims
    x = synth.host_x(w)
    T = x.shape[0]
    layers = []
    try:
        for layer in range(w.layers):
            layers.append(DeviceLayer(d, seed=layer, bias=synth.router_bias(w, layer)))
        ws = workspace(dims(d, 0), T)
        outs = [run_layer(lay, x, ws=ws) for lay in layers]  # back to back, every layer on the step's tokens
        for layer, (lay, (y, idx, _)) in enumerate(zip(layers, outs)):
            flips = check_selection(lay, x, idx)
            offsets = check_permutation(d, idx, ws=ws)
            sample = _subset(idx, offsets, 1024, d.n_experts)
            compare_layer(lay, x, y, idx, sample, nthreads=NCPU, what=f"prefill_32k layer {layer}")
            print(f"prefill_32k layer {layer}: {flips} boundary-tie tokens of {T}; {len(sample)} tokens compared")
            lay._experts_host.clear()
    finally:
        del layers
        torch.cuda.empty_cache()
