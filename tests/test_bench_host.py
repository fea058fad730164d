"""Host-side logic of bench.py on the CPU: byte accounting, clock parsing, and
the multi-rank timing reduction over a world-size-2 gloo group."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl


def test_prefill_bytes_match_the_stated_figure():
    # 4 x 4096 tokens, dim 8192: x + out = 2 x 268,435,456 B; states read and
    # written 4 x 8192 x 3 x 2 B each way; weight 65,536 B; bias 16,384 B.
    case = wl.varlen_prefill(1, [4096] * 4, 64, 4, num_cache_lines=4, has_init="all")
    dim = 8192
    want_big = 4 * dim * 16384 + 4 * dim * 3 * 2 * 2 + dim * 4 * 2 + dim * 2
    scaled = bench.prefill_bytes(case) - (4 * 5 + 4 * 4 + 4)  # drop index vectors
    assert scaled * (dim // 64) == want_big
    assert round(want_big / 1e6, 1) == 537.3


def test_decode_bytes_match_the_stated_figure():
    case = wl.decode(2, 256, 64, 4, num_lines=512)
    per_row = 64 * 2 * (1 + 1 + 3 + 3)
    assert bench.decode_bytes(case) == 256 * per_row + 64 * 4 * 2 + 64 * 2 + 4 * 256


def test_paged_bytes_count_cached_taps():
    # one decode token at position 10 (3 cached taps: positions 7, 8, 9 in
    # blocks 1, 2, 2 of size 4) and one prefill of 2 tokens starting at 0 (no
    # taps before position 0)
    case = wl.paged(3, [1, 2], [10, 0], H=1, ws=8, N=4, D=8, num_blocks=8, off_s=0)
    C, T = 8, 3
    want = 2 * T * C * 2 + 3 * C * 2 + 3 * C * 2 + C * 4 * 2 + T * 24 + 2 * 4 + 4 * 3
    assert bench.paged_bytes(case) == want


def test_paged_bytes_count_each_cached_position_once():
    # a 4-token spec request at position 10: its first three tokens read
    # 3 + 2 + 1 cached taps, but only positions 7, 8 and 9 (block-table
    # entries 1 and 2) need to be read
    case = wl.paged(4, [4], [10], H=1, ws=8, N=4, D=8, num_blocks=8, off_s=0)
    C, T = 8, 4
    want = 2 * T * C * 2 + 4 * C * 2 + 3 * C * 2 + C * 4 * 2 + T * 24 + 2 * 4 + 4 * 2
    assert bench.paged_bytes(case) == want


def test_clock_summary_flags_throttling():
    rows = [["2026/12/02 10:00:00.100", "1965", "2070", "900", "0x0", "Not Active",
             "Not Active", "Not Active", "Active"],
            ["2026/12/02 10:00:00.200", "1980", "2070", "910", "0x0", "Not Active",
             "Not Active", "Active", "Not Active"],
            ["garbage"]]
    s = bench.summarize_clocks([r for r in rows if len(r) >= 9])
    assert s["sm_mhz"] == pytest.approx(1972.5)
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier()
        seconds = 1.0 + rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(seconds)
        rate = bench.whole_job_rate(100.0, 10, world, worst)
        results[rank] = (worst, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        for r in range(2):
            worst, rate = results[r]
            assert worst == 2.0
            assert rate == pytest.approx(100.0 * 10 * 2 / 2.0)
