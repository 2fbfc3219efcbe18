"""Host-side logic of bench.py without a GPU: the replica aggregation over a
world-size-2 gloo group, interval bookkeeping and clock summaries."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    g = bench.init_group(world)
    bench.barrier(g)
    mx = bench.max_over_ranks(10.0 + rank, g)
    sm = bench.sum_over_ranks(100.0 * (rank + 1), g)
    out.put((rank, mx, sm))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_timing_takes_max_and_work_takes_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_single_process_needs_no_group():
    assert bench.init_group(1) is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.sum_over_ranks(2.0, None) == 2.0


class FakeEvent:
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_interval_stats_assigns_each_gap_to_the_call_that_ends_it():
    marks = [(FakeEvent(0.0), None, 0), (FakeEvent(1.0), "quant_w", 10), (FakeEvent(3.0), "fprop", 100),
             (FakeEvent(3.5), None, 0), (FakeEvent(4.0), "fprop", 100)]
    st = bench.interval_stats(marks)
    assert st["quant_w"] == [1, 1.0, 10]
    assert st["fprop"] == [2, 2.5, 200]


def test_clock_summary():
    rows = [{"sm": 1800.0, "sm_max": 2032.0, "power": 900.0, "active": []},
            {"sm": 1200.0, "sm_max": 2032.0, "power": 1100.0, "active": ["sw_power_cap"]},
            {"sm": 1500.0, "sm_max": 2032.0, "power": 1000.0, "active": ["sw_power_cap"]}]
    c = bench.summarise_clocks(rows)
    assert c["sm_mhz"] == 1500.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.summarise_clocks([])["samples"] == 0


def test_gemm_flops_counts_three_gemms_for_backward_linears():
    from blockwise_fp8_linear_quantise_b300 import workloads
    wl = workloads.make("stack28")
    specs = bench.linear_list(wl, 28)
    assert len(specs) == 112
    assert bench.gemm_flops(specs) == pytest.approx(138.54e12, rel=1e-3)
    assert len(bench.linear_list(wl, 1)) == 4
    assert bench.gemm_flops(bench.linear_list(workloads.make("mlp_gateup"), 28)) == 2 * 8192 * 12288 * 2048


def test_kernel_hash_ignores_comments_but_not_code():
    src = 'asm("mov.u32 %0, 1; // not a comment");  // a comment\nint x = 1; /* block */ int y = 2;'
    assert bench.strip_comments(src) == 'asm("mov.u32 %0, 1; // not a comment"); int x = 1; int y = 2;'
    assert bench.strip_comments(src.replace("// a comment", "// another one")) == bench.strip_comments(src)
    assert bench.strip_comments(src.replace("x = 1", "x = 2")) != bench.strip_comments(src)
    assert len(bench.kernel_source_hash()) == 16
