"""Benchmark of the routed-expert layer (one Stable-LatentMoE layer with MXFP4 experts).

  python bench.py [--workload decode_b1|decode_b64|prefill_4k|prefill_32k] [--steps K]
                  [--warmup W] [--gpus N] [--impl ours|reference]

A step is one k3moe_layer_run (on layers prepared once by k3moe_layer_init, timed apart as
``init_s``) over one batch of synthetic tokens (seeded generator, K3
shapes: hidden 7168, latent 3584, 896 experts of 17,547,264 bytes, top-16). Prints one JSON
line. ``value`` is device-timed throughput (CUDA events around exactly K steps, inputs
resident in HBM); ``e2e`` is the same through the C ABI with the step's tokens copied from
pinned host memory and its output copied back inside the timed region. Caches: the expert
store (15.7 GB) is far larger than L2, tokens are fresh every step, and the dense weights
rotate over 8 copies (923 MB) so no step finds them in L2.

The default run (decode_b1, one GPU) then measures the metric's other configurations in child
processes of their own (decode_b64, prefill_4k with bf16, MXFP8 and MXFP4 activations,
prefill_32k with bf16 and MXFP4, and prefill_32k with unbiased routing; a few steps each) and
summarises their lines under "workloads";
--no-secondary skips them.

--impl reference times the CPU oracle (plain C, double accumulation) on the host cores on a
bounded sample of the same workload; see cpu_sample().

Multi-GPU: the layer does not shard across GPUs in this build (replicas only): under torchrun
every rank runs its own replica on its own GPU and rank 0 reports the sum of tokens/s over
the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (decode b1/b64, prefill 4K/32K) + % of HBM / FP4 roofline"
ACTQ_NAME = {0: "bf16", 1: "mxfp8", 2: "mxfp4"}
DENSE_COPIES = 8


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"], "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], None, set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- algorithmic work
def algorithmic(d, T, distinct_experts, shared_width=0):
    """Bytes and flops one layer step must move / compute (dense weights once, each selected
    expert's bytes once, activations of the step; shared_width = n_shared x shared_inter, the
    stacked bf16 shared experts, read once)."""
    dense_w = 2 * (d.n_experts * d.hidden + 2 * d.latent * d.hidden) + 2 * 3 * shared_width * d.hidden
    act = 2 * T * d.hidden * 2 + T * d.n_experts * 4
    expert = distinct_experts * d.expert_bytes
    flops = 2 * T * (d.n_experts * d.hidden + 2 * d.latent * d.hidden) + \
        2 * T * d.top_k * 3 * d.latent * d.inter + 2 * T * 3 * shared_width * d.hidden
    return dense_w + expert + act, flops


def max_over_ranks(v, dist=None, device="cpu"):
    """The largest of every rank's v (a time: the job is as slow as its slowest rank)."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(steps, tokens_per_step, world, ms):
    """Whole-job throughput: the tokens every rank processed over the max-over-ranks time."""
    return steps * tokens_per_step * world / (ms / 1e3)


def measured_traffic(workload, kernel):
    """DRAM bytes per launch of a kernel from the committed ncu capture (profiles/traffic.json),
    or None when there is none or the kernel's sources have changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t["workloads"][workload][kernel]
        h = hashlib.sha256()
        for p in e["source_files"]:
            with open(os.path.join(ROOT, p), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != e["source_sha256"]:
            return None
        return e["traffic"]
    except (OSError, KeyError, ValueError):
        return None


# Many tokens with e4m3 activations: the library runs the experts with at most this many rows on
# the weights-on-N kernel ("expert_ffn_mma") and the others on the many-token kernels.
SMALL_EXPERT_ROWS = 8


def expert_split(idx, n_experts, T, actq):
    """(distinct experts, sorted rows) of the many-token kernels ("big") and of the small-expert
    kernel, from one step's selections; None where the library does not split."""
    if T < 65 or actq == 2:
        return None
    c = np.bincount(np.asarray(idx).ravel(), minlength=n_experts)
    big = c > SMALL_EXPERT_ROWS
    small = (c > 0) & ~big
    return {"big": (int(big.sum()), int(c[big].sum())), "small": (int(small.sum()), int(c[small].sum()))}


def kernel_cost(name, d, T, distinct, rows, actq, shared_width=0, split=None):
    """Algorithmic (bytes, flops, tensor dtype) of one launch of a profiled kernel: weights read
    once per launch, activations read and results written once. split (expert_split): the
    many-token expert kernels and the small-expert kernel each count their own experts and rows."""
    L, I, H, E = d.latent, d.inter, d.hidden, d.n_experts
    if split and name in ("expert_glu_mma", "expert_down_mma"):
        distinct, rows = split["big"]
    elif split and name == "expert_ffn_mma":
        distinct, rows = split["small"]
    glu_w = 2 * (d.gate_q_bytes + d.gate_s_bytes)
    down_w = d.down_q_bytes + d.down_s_bytes
    # activation bytes per value on the tensor-core expert path: bf16 as two e4m3 rows (2),
    # MXFP8 one e4m3 row (1), MXFP4 one row of packed e2m1 codes (0.5)
    P = {0: 2, 1: 1, 2: 0.5}[actq]
    mma = "fp4" if actq == 2 else "fp8"  # the block-scaled MMA kind's rate
    gemv = T < 33  # token-at-a-time dense projections below 33 tokens
    table = {
        # router logits fp32 + z bf16 (+ its f16 block-scaled copy on the GEMV path)
        "router_latent_in": (2 * (E + L) * H + 2 * T * H + 4 * T * E + 2 * T * L * (2 if gemv else 1),
                             2 * T * (E + L) * H, "bf16"),
        "latent_out": (2 * H * L + 2 * T * L + 2 * T * H, 2 * T * H * L, "bf16"),
        "expert_glu_gemv": (distinct * glu_w + rows * (2 * L + 4 * I), 4 * rows * L * I, None),
        "expert_down_gemv": (distinct * down_w + rows * (2 * I + 4 * L), 2 * rows * L * I, None),
        "expert_act_quant": (rows * 2 * L + rows * (P * L + L // 32), 0, None),
        "expert_glu_mma": (distinct * glu_w + rows * (P * L + L // 32) + rows * (P * I + I // 32),
                           4 * rows * L * I, mma),
        "expert_down_mma": (distinct * down_w + rows * (P * I + I // 32) + 4 * rows * L,
                            2 * rows * L * I, mma),
        # both passes in one launch (decode): the GLU output is written and read back once
        "expert_ffn_mma": (distinct * (glu_w + down_w) + rows * (P * L + L // 32) +
                           2 * rows * (P * I + I // 32) + 4 * rows * L, 6 * rows * L * I, mma),
        "combine": (rows * 4 * L + 2 * T * L, 0, None),
        # gate + up (fp32 out), GLU, down (fp32 out); S = n_shared x shared_inter
        "shared_experts": (2 * 3 * shared_width * H + 2 * T * H + 2 * 4 * T * shared_width +
                           (2 + 8) * T * shared_width + 2 * T * shared_width + 4 * T * H,
                           6 * T * shared_width * H, "bf16"),
    }
    return table.get(name, (None, 0, None))


def roofline(name, per_launch_ms, cost, pk):
    """Roofline entry of a kernel: HBM-bound unless its algorithmic flops at the tensor peak of
    its dtype take longer than its bytes at the copy bandwidth. fp8 (the block-scaled
    e2m1 x e4m3 MMA rate) = measured bf16 x 2, the nominal dense ratio (4.5 / 2.25 PFLOP/s);
    fp4 (kind::mxf4, e2m1 x e2m1) = measured bf16 x 6 (13.5 / 2.25 PFLOP/s)."""
    ratio = {"fp8": 2.0, "fp4": 6.0}
    kb, fl, dt = cost
    if not kb:
        return {"bound": "hbm", "kernel": name, "achieved": None, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": None, "traffic": None}
    t = per_launch_ms / 1e3
    tensor_peak = pk["bf16_tflops"] * ratio.get(dt, 1.0) if dt else None
    t_hbm = kb / (pk["hbm_gbs"] * 1e9)
    t_tc = fl / (tensor_peak * 1e12) if tensor_peak else 0.0
    if tensor_peak and t_tc > t_hbm:
        ach = fl / t / 1e12
        return {"bound": "tensor", "kernel": name, "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": ach / tensor_peak, "traffic": None,
                "peak_src": pk["src"] + " bf16 burst" + (f" x {ratio[dt]:g} ({dt} nominal ratio)" if dt in ratio else ""),
                "algorithmic_flops_per_launch": fl, "avg_launch_ms": per_launch_ms}
    ach = kb / t / 1e9
    return {"bound": "hbm", "kernel": name, "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "traffic": None, "peak_src": pk["src"] + " (burst copy)",
            "algorithmic_bytes_per_launch": kb, "avg_launch_ms": per_launch_ms,
            "tensor_frac": (fl / t / 1e12 / tensor_peak) if tensor_peak else None}


# ---------------------------------------------------------------- CPU oracle sample
def cpu_sample(w, layer_seed, x_np, idx_sample, units_per_step, steps, nthreads, pool=None, actq=0):
    """Times the oracle on (token, slot) units: each unit is one routed expert row through the
    oracle (gate/up, GLU, down; ~33M MACs) plus 1/k of that token's dense work (router, latent
    in and latent out rows), i.e. 1/k of a token. Units run on `nthreads` host threads. With
    `pool`, steps cycle through the first `pool` units only (the oracle decodes the weights on
    every call, so a repeated unit costs the same; fewer experts are generated on the host).
    Returns (layer, run_step)."""
    import oracle
    import synth

    d = w.dims
    k = d.top_k
    wr, wi, wo = synth.host_dense(d, layer_seed)
    experts = {}
    units = []
    for t in range(idx_sample.shape[0]):
        for j in range(k):
            e = int(idx_sample[t, j])
            units.append((t, j, e))
    if pool:
        units = units[:max(units_per_step, pool)]
    need = {e for (_, _, e) in units[: units_per_step * steps]}
    for e in need:
        experts[e] = synth.host_expert(d, layer_seed, e)
    lay = oracle.Layer(d, wr, wi, wo, experts, actq=actq)
    _, z_all = oracle.dense_proj(wi, x_np[: idx_sample.shape[0]])
    E_sl, L_sl, H_sl = d.n_experts // k, d.latent // k, d.hidden // k

    def run_unit(u):
        t, j, e = u
        xt = x_np[t:t + 1]
        oracle.dense_proj(wr[j * E_sl:(j + 1) * E_sl], xt)
        oracle.dense_proj(wi[j * L_sl:(j + 1) * L_sl], xt)
        lay.expert_row(e, z_all[t])
        oracle.dense_proj(wo[j * H_sl:(j + 1) * H_sl], z_all[t:t + 1])

    def step_units(s):
        """The units of step s: exactly units_per_step of them, cycling through the sample."""
        n = len(units)
        return [units[(s * units_per_step + i) % n] for i in range(units_per_step)]

    def run_step(s):
        us = step_units(s)
        ths = [threading.Thread(target=lambda grp=us[i::nthreads]: [run_unit(u) for u in grp])
               for i in range(min(nthreads, len(us)))]
        for th in ths:
            th.start()
        for th in ths:
            th.join()

    run_step.units = step_units
    return lay, run_step


# The other configurations the metric is quoted on, measured after the headline (decode_b1) in
# the default run, each in a child process of its own (its memory freed at exit) with a fixed
# number of steps; their lines are summarised under "workloads" of the one JSON line.
SECONDARY = (("decode_b64", 0, 100), ("prefill_4k", 0, 10), ("prefill_4k", 1, 10), ("prefill_4k", 2, 10),
             ("prefill_32k", 0, 3), ("prefill_32k_uniform", 0, 3), ("prefill_32k", 2, 3))


def summarize_line(line):
    """The figures of one bench JSON line that the headline line carries for it."""
    j = json.loads(line)
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "distinct_experts_last_step", "init_s")
    out = {k: j.get(k) for k in keep}
    out["e2e"] = j.get("e2e", {}).get("value")
    r = j.get("roofline") or {}
    out["roofline"] = {k: r.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit", "frac", "traffic")}
    out["step_frac_hbm"] = (j.get("step_roofline") or {}).get("frac_hbm")
    out["clocks"] = j.get("clocks")
    out["config"] = {k: (j.get("config") or {}).get(k) for k in ("workload", "tokens_per_step", "actq", "layers")}
    return out


def run_secondary(timeout_s=900):
    res = {}
    for wl, actq, steps in SECONDARY:
        key = wl + ("" if actq == 0 else "_" + ACTQ_NAME[actq])
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", wl, "--actq", str(actq), "--steps",
               str(steps), "--warmup", "3", "--no-cpu-baseline", "--no-secondary"]
        try:
            p = subprocess.run(cmd, capture_output=True, text=True, timeout=timeout_s)
            lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
            if p.returncode != 0 or not lines:
                res[key] = {"error": f"exit {p.returncode}: " + (p.stderr.strip().splitlines() or ["no output"])[-1][:300]}
            else:
                res[key] = summarize_line(lines[-1])
        except (subprocess.TimeoutExpired, OSError, ValueError) as e:
            res[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return res


def run_reference(args, w):
    """Reference arm: the CPU oracle on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    nth = os.cpu_count() or 1
    d = w.dims
    T = min(w.x_count, 64)  # sample tokens (decode_b1 draws them from its 1000 fresh tokens)
    x = synth.host_x(w, 0, T)
    import oracle
    wr, _, _ = synth.host_dense(d, 0)
    idx = oracle.select_topk(oracle.router_logits_np(x, wr, synth.router_bias(w)), d.top_k)
    # per-step sample sized so warmup + steps stay within ~150 s of wall time, calibrated on
    # one unit (a step never takes less than one unit's time)
    _, step1 = cpu_sample(w, 0, x, idx, 1, 1, 1)
    t0 = time.perf_counter()
    step1(0)
    per_unit_s = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    units = max(1, min(nth * 64, int(budget * nth / per_unit_s)))
    units = max(1, (units // nth) * nth) if units >= nth else units
    _, step = cpu_sample(w, 0, x, idx, units, args.steps + args.warmup, nth)
    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s)
    el = time.perf_counter() - t0
    nl = max(1, int(getattr(w, "layers", 1) or 1))
    tokens = args.steps * units / d.top_k  # every step runs exactly `units` units
    val = tokens / el / nl  # through the whole stack of layers
    sample = (f"{units} (token, expert-slot) units per step = {units / d.top_k:.3g} tokens through one "
              f"layer of the {w.name} workload, cycling over the {T * d.top_k} units of {T} sample tokens "
              f"(expert row + 1/{d.top_k} of the token's dense rows each; tokens/s divided by its {nl} layer(s))")
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
           "config": {"workload": w.name, "tokens_per_step": w.tokens, "layers": nl},
           "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------- GPU arm
def run_ours(args, w):
    import torch
    import mxfp4_expert_ffn_top16_gb300 as k3
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    d = w.dims
    T = w.tokens
    E = d.n_experts

    # --- layers: one layer = one expert store with DENSE_COPIES copies of its dense weights;
    # a stack of n layers (independent seeded weights, run back to back) = n stores, one dense
    # set each (together already far larger than L2)
    t_setup = time.time()
    nl = max(1, int(getattr(w, "layers", 1) or 1))
    sizes = {"gate_q": E * d.gate_q_bytes, "gate_s": E * d.gate_s_bytes, "up_q": E * d.gate_q_bytes,
             "up_s": E * d.gate_s_bytes, "down_q": E * d.down_q_bytes, "down_s": E * d.down_s_bytes}
    ns, si = (2, args.shared_inter) if args.shared_inter else (0, 0)
    S = ns * si
    dims = k3.Dims(d.hidden, d.latent, d.inter, d.n_experts, d.top_k, 0, args.actq, ns, si)
    shw = {n: torch.empty(S * d.hidden, dtype=torch.int16, device=dev) for n in ("w_sgate", "w_sup", "w_sdown")}
    if S:
        synth.dev_fill_shared(d, ns, si, 0, {n: t.data_ptr() for n, t in shw.items()}, sh)
    shp = [shw[n].data_ptr() if S else None for n in ("w_sgate", "w_sup", "w_sdown")]
    if nl > 1:
        keep = []
        wts = []
        for layer in range(nl):
            exl = {n: torch.empty(b, dtype=torch.uint8, device=dev) for n, b in sizes.items()}
            ddl = {"w_router": torch.empty(E * d.hidden, dtype=torch.int16, device=dev),
                   "w_in": torch.empty(d.latent * d.hidden, dtype=torch.int16, device=dev),
                   "w_out": torch.empty(d.hidden * d.latent, dtype=torch.int16, device=dev)}
            pl = {n: t.data_ptr() for n, t in exl.items()}
            pl.update({n: t.data_ptr() for n, t in ddl.items()})
            synth.dev_fill_layer(d, layer, pl, sh)
            bl = synth.router_bias(w, layer)
            bt = None if bl is None else torch.from_numpy(bl).to(dev)
            keep.append((exl, ddl, bt))
            wts.append(k3.Weights(ddl["w_router"].data_ptr(), None if bt is None else bt.data_ptr(),
                                  ddl["w_in"].data_ptr(), ddl["w_out"].data_ptr(),
                                  *[exl[n].data_ptr() for n in ("gate_q", "gate_s", "up_q", "up_s",
                                                                "down_q", "down_s")], *shp))
    ex = {n: torch.empty(b if nl == 1 else 0, dtype=torch.uint8, device=dev) for n, b in sizes.items()}
    dense = []
    for c in range(DENSE_COPIES if nl == 1 else 0):
        dd = {"w_router": torch.empty(E * d.hidden, dtype=torch.int16, device=dev),
              "w_in": torch.empty(d.latent * d.hidden, dtype=torch.int16, device=dev),
              "w_out": torch.empty(d.hidden * d.latent, dtype=torch.int16, device=dev)}
        dense.append(dd)
    bias_np = synth.router_bias(w)
    if nl == 1:
        ptrs = {n: t.data_ptr() for n, t in ex.items()}
        ptrs.update({n: t.data_ptr() for n, t in dense[0].items()})
        synth.dev_fill_layer(d, 0, ptrs, sh)
        for c in range(1, DENSE_COPIES):
            for n in dense[c]:
                dense[c][n].copy_(dense[0][n])
        bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
        wts = [k3.Weights(dd["w_router"].data_ptr(), None if bias is None else bias.data_ptr(),
                          dd["w_in"].data_ptr(), dd["w_out"].data_ptr(),
                          *[ex[n].data_ptr() for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q",
                                                       "down_s")], *shp) for dd in dense]
    nx = w.x_count
    x = torch.empty((nx, d.hidden), dtype=torch.int16, device=dev)
    synth.dev_fill_x(w, x.data_ptr(), cuda_stream=sh)
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=dev)
    hbuf = [torch.empty((T, d.hidden), dtype=torch.int16, device=dev) for _ in range(2 if nl > 1 else 0)]
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=dev)
    nbytes = k3.k3moe_workspace_size(dims, T)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup
    # prepared layers (the expert scales repacked once for the decode kernel): outside every
    # timed region, reported as init_s
    t_init = time.time()
    handles = [k3.k3moe_layer_init(dims, wt, sh) for wt in wts] if args.prepare else None
    init_s = time.time() - t_init
    nsteps_x = max(1, nx // T)

    cur = {"stream": sh}  # the stream the layer calls go to (a capture stream while recording a graph)

    def step(i, xp=None, yp=None):
        xi = xp if xp is not None else x[(i % nsteps_x) * T:].data_ptr()
        yo = yp or y.data_ptr()
        if nl == 1:
            if handles:
                k3.k3moe_layer_run(handles[i % DENSE_COPIES], xi, T, yo, idx.data_ptr(), None, ws.data_ptr(), nbytes,
                                   cur["stream"])
            else:
                k3.k3moe_layer_forward(dims, wts[i % DENSE_COPIES], xi, T, yo, idx.data_ptr(), None,
                                       ws.data_ptr(), nbytes, cur["stream"])
            return
        # every layer takes the step's tokens (chaining the synthetic layers' outputs would
        # overflow within a few layers: the random experts amplify the activations)
        for layer in range(nl):
            dst = yo if layer == nl - 1 else hbuf[layer % 2].data_ptr()
            if handles:
                k3.k3moe_layer_run(handles[layer], xi, T, dst, idx.data_ptr(), None, ws.data_ptr(), nbytes,
                                   cur["stream"])
            else:
                k3.k3moe_layer_forward(dims, wts[layer], xi, T, dst, idx.data_ptr(), None, ws.data_ptr(),
                                       nbytes, cur["stream"])

    def capture(G):
        """A CUDA graph of G consecutive steps (the layer calls neither allocate nor synchronise,
        so they capture as they are, programmatic-launch edges included); None if capture fails."""
        try:
            g = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream()
            cs.wait_stream(stream)
            with torch.cuda.graph(g, stream=cs):
                cur["stream"] = cs.cuda_stream
                for j in range(G):
                    step(args.warmup + j)
            stream.wait_stream(cs)
            return g
        except Exception as e:  # fall back to stream launches
            print(f"bench: graph capture failed ({e}); timing stream launches", file=sys.stderr)
            return None
        finally:
            cur["stream"] = sh

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
            torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    st = k3.k3moe_check(ws.data_ptr(), sh)
    if st != 0:
        raise RuntimeError("warmup: " + k3.status_string(st))

    # --- pass 1: device-timed value: exactly K steps, replayed from a CUDA graph of G captured
    # steps (G the largest divisor of K up to --graph-steps; tokens cycle over G sets) or, with
    # --graph-steps 0, launched step by step
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    G = min(args.graph_steps, args.steps)
    while G > 1 and args.steps % G:
        G -= 1
    graph = capture(G) if G >= 1 and args.graph_steps > 0 else None
    if graph is not None:
        graph.replay()  # untimed: the first replay uploads the graph
        barrier()
        ev0.record(stream)
        for r in range(args.steps // G):
            graph.replay()
    else:
        barrier()
        ev0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
    ev1.record(stream)
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    st = k3.k3moe_check(ws.data_ptr(), sh)
    if st != 0:
        raise RuntimeError("timed: " + k3.status_string(st))
    idx_last = idx.cpu().numpy()
    distinct = int(len(np.unique(idx_last)))
    split = expert_split(idx_last, E, T, args.actq)

    # --- pass 2: the same steps with per-kernel CUDA events (roofline of the top kernel)
    barrier()
    k3.k3moe_profile(1)
    for i in range(args.steps):
        step(args.warmup + i)
    prof = k3.k3moe_profile(0)
    barrier()

    # --- pass 3: end to end through the C ABI with pinned host buffers
    xh = torch.empty((nx, d.hidden), dtype=torch.int16, pin_memory=True)
    xh.copy_(x.cpu())
    yh = torch.empty((args.steps, T, d.hidden), dtype=torch.int16, pin_memory=True)
    xs = torch.empty((T, d.hidden), dtype=torch.int16, device=dev)
    # one layer on a prepared handle: k3moe_layer_run_host takes the pinned buffers themselves (its
    # own kernels read the tokens from and write the output to host memory); otherwise copies
    # from and to pinned memory around each layer call
    host_call = bool(handles) and nl == 1
    barrier()
    ev0.record(stream)
    for i in range(args.steps):
        j = (args.warmup + i) % nsteps_x
        if host_call:
            k3.k3moe_layer_run_host(handles[(args.warmup + i) % DENSE_COPIES], xh[j * T:(j + 1) * T].data_ptr(), T,
                                    yh[i].data_ptr(), idx.data_ptr(), None, ws.data_ptr(), nbytes, cur["stream"])
        else:
            xs.copy_(xh[j * T:(j + 1) * T], non_blocking=True)
            step(args.warmup + i, xp=xs.data_ptr())
            yh[i].copy_(y, non_blocking=True)
    ev1.record(stream)
    barrier()
    ms_e2e = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    clk = clocks.stop()

    value = job_tokens_per_s(args.steps, T, world, ms)
    e2e = job_tokens_per_s(args.steps, T, world, ms_e2e)
    pk = peaks()
    # dominant kernel by time share
    top = max(prof.items(), key=lambda kv: kv[1][0])
    name, (tot_ms, launches) = top
    per_launch_ms = tot_ms / max(1, launches)
    step_bytes, step_flops = algorithmic(d, T, distinct, S)
    step_bytes, step_flops = step_bytes * nl, step_flops * nl  # every layer of the stack
    kernels_per_step = {"permute": 1 if T <= 256 else 3}
    launches_total = sum(n for _, n in prof.values()) + \
        (kernels_per_step["permute"] - 1) * prof.get("permute", (0, 0))[1]
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4 weights x " + ACTQ_NAME[args.actq] + " activations, fp32 accumulate",
        "data": "synthetic (seeded SplitMix64; bf16 ~N(0,1) tokens, ~N(0,0.02) dense, U{0..15} codes, U{120..127} e8m0)",
        "config": {"workload": w.name, "tokens_per_step": T, "hidden": d.hidden, "latent": d.latent,
                   "inter": d.inter, "n_experts": d.n_experts, "top_k": d.top_k,
                   "router_bias": w.bias, "actq": ACTQ_NAME[args.actq], "layers": nl,
                   "l2": ("expert store 15.7 GB >> L2; fresh tokens per step; dense weights rotate over 8 copies"
                          if nl == 1 else f"{nl} layers with independent weights ({nl * 15.7:.0f} GB of experts) run back to "
                          "back on the same tokens; fresh tokens per step"),
                   "parallelism": f"replicas x{world}",
                   "launch": (f"value: CUDA graph of {G} captured steps replayed {args.steps // G} times "
                              f"(tokens cycle over {G} sets); per-kernel and e2e passes: stream launches"
                              if graph is not None else "stream launches (programmatic dependent launch)"),
                   "shared_experts": (f"{ns} x {si} bf16 (width a parameter; not in the headline configuration)"
                                      if S else "none")},
        "roofline": roofline(name, per_launch_ms, kernel_cost(name, d, T, distinct, T * d.top_k, args.actq, S, split), pk),
        # (traffic filled in below from the committed capture of this workload, bf16 mode only)
        "step_roofline": {"algorithmic_bytes": step_bytes, "flops": step_flops,
                          "achieved_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
                          "frac_hbm": step_bytes / (ms / args.steps / 1e3) / 1e9 / pk["hbm_gbs"]},
        "kernels": {n: dict(ms_per_launch=(t / c if c else None), launches=c,
                            share=t / sum(v[0] for v in prof.values()),
                            frac=roofline(n, t / max(1, c), kernel_cost(n, d, T, distinct, T * d.top_k, args.actq, S, split),
                                          pk)["frac"]) for n, (t, c) in prof.items() if c},
        "distinct_experts_last_step": distinct,
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": T * d.hidden * 2,
                "d2h_bytes_per_step": T * d.hidden * 2,
                "call": ("k3moe_layer_run_host on pinned host buffers (the library's kernels read the tokens "
                         "and write the output over the CPU-GPU link)" if host_call else
                         "pinned-memory copies around each layer call")},
        "gpu_launches": int(launches_total / max(1, 1)),
        "clocks": clk,
        "setup_s": setup_s,
        "init_s": init_s if handles else None,
    }
    for h in handles or []:
        k3.k3moe_layer_free(h)
    handles = None
    out["gpu_launches"] = int(launches_total)
    if not args.actq and not args.experts:
        out["roofline"]["traffic"] = measured_traffic(w.name, name)
    if rank == 0 and not args.no_cpu_baseline:
        nth = os.cpu_count() or 1
        xs_np = synth.host_x(w, 0, min(T, 8) if T > 1 else 16)
        import oracle
        wr, _, _ = synth.host_dense(d, 0)
        isamp = oracle.select_topk(oracle.router_logits_np(xs_np, wr, bias_np), d.top_k)
        # bounded sample: about 10 s of oracle work, calibrated on one step of nth units
        units = nth
        _, cstep = cpu_sample(w, 0, xs_np, isamp, units, 64, nth, pool=2 * nth, actq=args.actq)
        t0 = time.perf_counter()
        cstep(0)
        per_step = max(1e-3, time.perf_counter() - t0)
        steps_cpu = int(max(1, min(400, 10.0 / per_step)))
        t0 = time.perf_counter()
        for s in range(steps_cpu):
            cstep(1 + s)
        el = time.perf_counter() - t0
        out["cpu_baseline"] = {
            "value": steps_cpu * units / d.top_k / el / nl, "unit": "tokens/s", "cores": nth,
            "kind": "oracle",
            "sample": f"{steps_cpu * units} (token, expert-slot) units = {steps_cpu * units / d.top_k:.2f} "
                      f"tokens through one layer of {w.name} (tokens/s divided by its {nl} layer(s)); each "
                      f"unit = one expert row + 1/{d.top_k} of the token's dense rows, {el:.1f} s on {nth} threads"}
    if dist is not None:
        dist.destroy_process_group()
    return out if rank == 0 else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_b1")
    ap.add_argument("--actq", type=int, default=0, choices=[0, 1, 2],
                    help="activations: 0 bf16 (the headline), 1 MXFP8, 2 MXFP4 (kind::mxf4 experts)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prepare", dest="prepare", action="store_false",
                    help="call k3moe_layer_forward instead of k3moe_layer_run on layers prepared once by "
                         "k3moe_layer_init (scales repacked for the decode expert kernel)")
    ap.add_argument("--graph-steps", type=int, default=8,
                    help="steps per captured CUDA graph for the device-timed value (0: launch step by step)")
    ap.add_argument("--shared-inter", type=int, default=0,
                    help="also run two always-on bf16 shared experts of this width (their width is not "
                         "on the pages; the headline metric is the routed layer without them)")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="decode_b1 only: skip the runs of decode_b64, prefill_4k (bf16, MXFP8 and MXFP4 "
                         "activations) and prefill_32k (bf16 with Zipf and with unbiased routing, MXFP4) "
                         "that the default run adds under \"workloads\"")
    ap.add_argument("--experts", type=int, default=None,
                    help="profiling aid: the same workload with fewer experts (fits an ncu capture); "
                         "not a bench configuration")
    args = ap.parse_args()
    import dataclasses
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.experts:
        w = dataclasses.replace(w, dims=dataclasses.replace(w.dims, n_experts=args.experts))
    default_steps = {"decode_b1": 1000, "decode_b64": 200, "prefill_4k": 20, "prefill_32k": 4, "prefill_32k_uniform": 4}
    if args.steps is None:
        args.steps = default_steps.get(w.name, 20)
    if args.warmup is None:
        args.warmup = max(3, min(20, args.steps // 10))
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args, w)
        return
    out = run_ours(args, w)
    if out is None:
        return
    if out["n_gpus"] == 1 and args.secondary and w.name == "decode_b1" and not args.experts:
        # the headline's device memory is released (run_ours has returned) before the children
        # run; nothing of this process runs on the GPU meanwhile
        import torch
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        out["workloads"] = run_secondary()
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
