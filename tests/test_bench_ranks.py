"""The bench's multi-rank host logic on CPU: max-over-ranks timing across two gloo ranks on
127.0.0.1, the whole-job throughput, and the reference arm's non-zero ranks exiting without
work. (The GPU arm runs replicas: no collective on the data path.)"""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")  # rank 1 is the slow one
        q.put((rank, ms, bench.job_tokens_per_s(100, 64, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time, and the job throughput counts both ranks' tokens
    assert [o[1] for o in out] == [15.0, 15.0]
    assert all(abs(o[2] - 100 * 64 * 2 / 0.015) < 1e-6 for o in out)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_tokens_per_s(1000, 1, 1, 100.0) == 10000.0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_cpu_sample_steps_run_exactly_their_units():
    """The oracle sample that the reference arm and the cpu_baseline time: every step runs
    exactly units_per_step (token, slot) units, cycling through the sample when it is smaller,
    so the throughput counts the work that actually ran."""
    import numpy as np
    import oracle
    import synth
    w = synth.WORKLOADS["tiny"]
    d = w.dims
    x = synth.host_x(w, 0, 3)
    wr, _, _ = synth.host_dense(d, 0)
    idx = oracle.select_topk(oracle.router_logits_np(x, wr, None), d.top_k)  # 3 tokens x 4 slots = 12 units
    for per_step in (5, 12, 50):
        lay, step = bench.cpu_sample(w, 0, x, idx, per_step, 4, 2)
        calls = []
        real = lay.expert_row
        lay.expert_row = lambda e, z: (calls.append(e), real(e, z))[1]
        for s in range(3):
            assert len(step.units(s)) == per_step
            step(s)
        assert len(calls) == 3 * per_step
        flat = [u for s in range(3) for u in step.units(s)]
        n = len(idx.ravel())
        assert [u[2] for u in flat] == [int(idx.ravel()[i % n]) for i in range(3 * per_step)]
