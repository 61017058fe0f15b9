"""The benchmark's multi-rank path on the CPU: two gloo ranks run as replicas.

Each rank times its own steps; the job's time is the slowest rank's and its
throughput counts the tokens of every rank (weak scaling, no data exchange).
The reference arm does its work on rank 0 only; other ranks return nothing."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, per_rank_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        q.put((rank, bench.combine_ranks(per_rank_ms[rank], 8192, 10, dist)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    per_rank_ms = [10.0, 15.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, per_rank_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        ms_step, value = got[r]
        assert ms_step == pytest.approx(1.5)                       # 15 ms / 10 steps, the slower rank
        assert value == pytest.approx(2 * 8192 / 1.5e-3)           # both ranks' tokens over that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms_step, value = bench.combine_ranks(12.0, 4096, 4)
    assert ms_step == pytest.approx(3.0) and value == pytest.approx(4096 / 3e-3)


def test_reference_arm_only_on_rank_zero():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus, tokens, cpu_tokens = 1, 0, 2, 8192, 16
    assert bench.run_reference(Args(), rank=1, world=2) is None


def test_clock_summary_keeps_the_timed_region():
    """Samples outside [mark_start, mark_end] are dropped; throttle reasons
    seen inside are reported (host-side parsing only, no nvidia-smi)."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(None)
    idle = "1200, 2070, 150.0, 0x1, Not Active, Not Active, Not Active, Not Active"
    busy = "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"
    c.lines = [(0.0, idle), (1.0, busy), (1.1, capped), (1.2, busy), (2.0, idle)]
    c.t_start, c.t_end = 0.5, 1.5
    s = c.summary()
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    c.t_start, c.t_end = 5.0, 6.0  # nothing inside: every sample is summarised
    s = c.summary()
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 5
