"""The N > 1 path of bench.py on CPU: two gloo ranks in child processes.

Rows are independent (one replica of the workload per rank, no exchange step), so the only
cross-rank work is a barrier around the timed region and the max over ranks of the step time;
the whole-job value is all ranks' rows over that max.  The reference arm prints on rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = [3.0, 5.0][rank]                         # rank 1 is the slow one
        ms_max = bench.max_over_ranks_of(ms, world)
        value = bench.whole_job_rows_per_s(131072, ms_max, world)
        args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world, "batch": 8})()
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(args, rank)       # non-zero ranks return without work
        bench.rank_barrier(world)
        q.put((rank, ms_max, value, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(2):
        rank, ms_max, value, printed = q.get(timeout=120)
        out[rank] = (ms_max, value, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 5.0              # every rank sees the slowest rank's time
    assert out[0][1] == out[1][1] == pytest.approx(2 * 131072 / 5e-3)
    assert out[1][2] == ""                           # the reference arm prints on rank 0 only


class _StubStep:
    """Stands in for the GPU step in bench.run_steps: each step sleeps 2 ms x (rank + 1),
    so rank 1 is the slow one, and the workload's first values are kept to show which
    seed this rank drew."""

    def __init__(self, args, wl, rank, world):
        self.rank = rank
        self.fingerprint = wl.index_qk[0, 0, :8].tolist()
        self.steps = 0

    def step(self):
        import time
        time.sleep(0.002 * (self.rank + 1))
        self.steps += 1

    def sync(self):
        pass

    def check(self):
        pass

    def sampler(self):
        from contextlib import nullcontext
        return nullcontext(type("C", (), {"summary": staticmethod(lambda: {"stub": True})})())

    def time_steps(self, K):
        import time
        t = time.perf_counter()
        for _ in range(K):
            self.step()
        return 1e3 * (time.perf_counter() - t)

    def after_timed(self, args, world):
        return {"after": self.rank}

    def report(self, args, world, ms_step, after, clocks):
        return {"gpu_launches": 0, "stub": {"rank": self.rank, "fingerprint": self.fingerprint,
                                            "steps_run": self.steps, "after": after, "clocks": clocks}}


def _run_steps_rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        args = type("A", (), {"steps": 5, "warmup": 3, "gpus": world, "batch": 1})()
        buf = io.StringIO()
        with redirect_stdout(buf):
            line = bench.run_steps(args, rank, world, _StubStep)
        wl = bench.rank_workload(1, rank)
        q.put((rank, line, buf.getvalue(), wl.index_qk[0, 0, :8].tolist()))
    finally:
        dist.destroy_process_group()


def test_run_steps_two_gloo_ranks_seeds_reduction_and_one_line():
    """bench.run_steps, the skeleton of every bench run, under two gloo ranks with a
    stubbed device step: each rank draws its own seed, the step time is the slowest
    rank's, and rank 0 alone prints one line with n_gpus = 2."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_run_steps_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(2):
        rank, line, printed, fp = q.get(timeout=180)
        out[rank] = (line, printed, fp)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    line0, printed0, fp0 = out[0]
    line1, printed1, fp1 = out[1]
    assert line1 is None and printed1 == ""                  # rank 1 prints nothing
    lines = [l for l in printed0.splitlines() if l.strip()]
    assert len(lines) == 1 and json.loads(lines[0]) == line0
    assert line0["n_gpus"] == 2 and line0["steps"] == 5 and line0["warmup"] == 3
    # seeds: rank r draws seed 4 + r; the step ran on rank 0's own draw
    assert bench.rank_seed(0) == 4 and bench.rank_seed(1) == 5
    assert fp0 == workloads.scoring("bf16", seed=4, B=1).index_qk[0, 0, :8].tolist()
    assert fp1 == workloads.scoring("bf16", seed=5, B=1).index_qk[0, 0, :8].tolist()
    assert fp0 != fp1
    assert line0["stub"]["fingerprint"] == fp0 and line0["stub"]["steps_run"] == 3 + 5
    # the slowest rank's time (rank 1 sleeps 4 ms a step) decides; value = all rows / that time
    assert line0["ms_per_step"] >= 4.0
    assert line0["value"] == pytest.approx(2 * 16384 / (line0["ms_per_step"] * 1e-3))
    assert line0["config"] == bench.step_config(1, 16384, 4096)
    assert line0["stub"]["clocks"] == {"stub": True} and line0["scaling"] == "weak"


def test_reference_arm_times_whole_oracle_steps_with_the_same_config():
    """--impl reference on one sequence, one step: whole oracle steps (not extrapolated),
    and the same config dict the GPU arm prints."""
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 1, "batch": 1})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, 0)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["extrapolated"] is False
    assert line["config"] == bench.step_config(1, 16384, 4096)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["sample"].startswith("whole steps")
    assert line["value"] == pytest.approx(16384 / (line["ms_per_step"] * 1e-3))


def test_oracle_full_step_equals_the_oracle_called_whole():
    """The reference arm's threaded slabs compute what one call of each oracle function
    over the whole (small) workload computes."""
    sys.path.insert(0, ROOT)
    import concurrent.futures as cf
    import numpy as np
    import bench
    import oracle
    import workloads
    wl = workloads.custom(2, 1100, [1100, 613], seed=7)
    B, S, NB = wl.B, wl.S, wl.num_blocks
    logits = np.empty((B * S, NB), np.float32)
    with cf.ThreadPoolExecutor(4) as pool:
        bench.oracle_full_step(wl, pool, 4, logits)
    q = oracle.q_prep("bf16", wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_q, wl.eps)
    kb = oracle.k_compress("bf16", wl.index_qk, wl.cos_sin, wl.context_lengths, wl.w_k, wl.eps, NB, 0, NB, 0)
    ref = oracle.scores("bf16", q, kb, wl.context_lengths)
    assert np.array_equal(logits.view(np.uint32), ref.view(np.uint32))


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks_of(2.5, 1) == 2.5
    assert bench.whole_job_rows_per_s(1000, 2.0, 1) == pytest.approx(5e5)
    json.dumps({"v": bench.whole_job_rows_per_s(1, 1.0, 4)})


def test_k2_traffic_profile_matches_the_kernel_source():
    """The bench line's roofline traffic comes from the committed K2 ncu summary, which
    records the hash of the K2 source it was captured on: the two must still agree, the
    figure reported must be the one recorded, and it must be close to K2's algorithmic bytes
    at B=8 (a little below them: the last logits are still dirty in L2 when the kernel ends)."""
    sys.path.insert(0, ROOT)
    import re
    import bench
    got = bench.k2_profiled_traffic(8)
    assert got is not None, "the K2 ncu summary was captured on another K2 source: recapture it"
    with open(os.path.join(ROOT, "profiles", "k2_scores_tc_B4_S16384.md")) as f:
        want = int(re.search(r"traffic_bytes_per_launch_B8: (\d+)", f.read()).group(1))
    assert got == want
    alg = bench.algorithmic_bytes(np.full(8, 16384, np.int32), 8, 16384, 4096)["k2"]
    assert 0.9 * alg <= got <= 1.05 * alg
