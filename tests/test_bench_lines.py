"""The bench's summary of the secondary configurations (host logic, no GPU): what one child's
JSON line is reduced to, and a failing child recorded as an error instead of ending the run."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _line():
    return json.dumps({
        "metric": bench.METRIC, "value": 537900.0, "unit": "tokens/s", "ms_per_step": 7.61, "steps": 10,
        "warmup": 3, "dtype": "mxfp4 weights x bf16 activations, fp32 accumulate",
        "distinct_experts_last_step": 870, "init_s": 0.004,
        "e2e": {"value": 495900.0, "unit": "tokens/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1},
        "roofline": {"kernel": "expert_glu_mma", "bound": "hbm", "achieved": 2410.0, "peak": 6800.7,
                     "unit": "GB/s", "frac": 0.354, "traffic": None, "extra": 1},
        "step_roofline": {"frac_hbm": 0.30},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
        "config": {"workload": "prefill_4k", "tokens_per_step": 4096, "actq": "bf16", "layers": 1, "hidden": 7168},
    })


def test_summary_keeps_the_figures_and_drops_the_rest():
    s = bench.summarize_line(_line())
    assert s["value"] == 537900.0 and s["ms_per_step"] == 7.61 and s["steps"] == 10 and s["warmup"] == 3
    assert s["e2e"] == 495900.0
    assert s["roofline"]["frac"] == 0.354 and s["roofline"]["kernel"] == "expert_glu_mma"
    assert "extra" not in s["roofline"]
    assert s["step_frac_hbm"] == 0.30
    assert s["clocks"]["sm_mhz"] == 2070.0
    assert s["config"] == {"workload": "prefill_4k", "tokens_per_step": 4096, "actq": "bf16", "layers": 1}


def test_children_commands_and_a_failing_child(monkeypatch):
    seen = []

    def fake_run(cmd, capture_output, text, timeout):
        seen.append(cmd)
        wl = cmd[cmd.index("--workload") + 1]
        if wl.startswith("prefill_32k"):
            return subprocess.CompletedProcess(cmd, 1, "", "Traceback ...\nRuntimeError: out of memory\n")
        return subprocess.CompletedProcess(cmd, 0, "log line\n" + _line() + "\n", "")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    res = bench.run_secondary()
    assert set(res) == {"decode_b64", "prefill_4k", "prefill_4k_mxfp8", "prefill_4k_mxfp4", "prefill_32k",
                        "prefill_32k_uniform", "prefill_32k_mxfp4"}
    assert res["prefill_32k"] == {"error": "exit 1: RuntimeError: out of memory"}
    assert res["prefill_32k_mxfp4"] == {"error": "exit 1: RuntimeError: out of memory"}
    assert res["prefill_32k_uniform"] == {"error": "exit 1: RuntimeError: out of memory"}
    assert res["prefill_4k"]["value"] == 537900.0
    for cmd in seen:  # every child: its own workload, at least 3 warm-up steps, no recursion
        assert "--no-secondary" in cmd and "--no-cpu-baseline" in cmd
        assert int(cmd[cmd.index("--warmup") + 1]) >= 3
    actq = {c[c.index("--workload") + 1] + c[c.index("--actq") + 1] for c in seen}
    assert actq == {"decode_b640", "prefill_4k0", "prefill_4k1", "prefill_4k2", "prefill_32k0", "prefill_32k2",
                    "prefill_32k_uniform0"}


def test_expert_split_counts_big_and_small_experts():
    import numpy as np
    # 80 tokens, top-2: expert 0 gets every token (80 rows), expert 1 the first 6 tokens, expert 2
    # the next 9, expert 3 the rest (65)
    idx = np.zeros((80, 2), np.int32)
    idx[:6, 1] = 1
    idx[6:15, 1] = 2
    idx[15:, 1] = 3
    s = bench.expert_split(idx, 5, 80, 0)
    assert s == {"big": (3, 80 + 9 + 65), "small": (1, 6)}
    assert bench.expert_split(idx, 5, 64, 0) is None   # the decode kernels take every expert
    assert bench.expert_split(idx, 5, 80, 2) is None   # MXFP4 activations: no split
    # the split changes which experts each kernel is charged for
    import synth
    d = synth.K3
    full = bench.kernel_cost("expert_glu_mma", d, 80, 4, 160, 0)
    big = bench.kernel_cost("expert_glu_mma", d, 80, 4, 160, 0, split=s)
    small = bench.kernel_cost("expert_ffn_mma", d, 80, 4, 160, 0, split=s)
    assert big[0] < full[0] and small[0] > 0 and big[1] == 4 * 154 * d.latent * d.inter
