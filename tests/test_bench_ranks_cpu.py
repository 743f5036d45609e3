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
        args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world})()
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


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks_of(2.5, 1) == 2.5
    assert bench.whole_job_rows_per_s(1000, 2.0, 1) == pytest.approx(5e5)
    json.dumps({"v": bench.whole_job_rows_per_s(1, 1.0, 4)})


def test_k2_traffic_profile_matches_the_kernel_source():
    """The bench line's roofline traffic comes from the committed K2 ncu summary, which
    records the hash of the K2 source it was captured on: the two must still agree."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.k2_profiled_traffic(8) == 2168935424
