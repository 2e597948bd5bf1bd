"""Host logic of bench.py on the CPU: the max-over-ranks timing and the
whole-job aggregate with two gloo ranks, the roofline arithmetic, the
per-launch statistics and the nvidia-smi clock parser."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier()
        # rank r "took" 1 + r seconds: every rank sees the slowest one
        t = bench.reduce_max(1.0 + rank)
        v = bench.aggregate(100.0, world, t)
        out.put((rank, t, v))
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, v in res:
        assert t == 2.0                    # the slower rank's time
        assert v == 100.0 * 2 / 2.0        # units of all ranks / that time


def test_single_process_helpers_are_identities():
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier()
    assert bench.aggregate(10.0, 1, 2.0) == 5.0


def test_roofline_picks_the_slower_bound():
    # 1 GB at 1000 GB/s = 1 ms; 1 TFLOP at 2000 TFLOP/s = 0.5 ms -> HBM bound
    r = bench.roofline(1e9, 1e12, 2e-3, 1000.0, 2000.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(500.0)
    assert r["frac"] == pytest.approx(0.5)
    # tensor bound when the flops take longer
    r = bench.roofline(1e9, 4e12, 4e-3, 1000.0, 2000.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(0.5)
    assert r["t_mem_us"] == pytest.approx(1000.0) and r["t_tensor_us"] == pytest.approx(2000.0)


def test_step_stats():
    s = bench.step_stats([3.0, 1.0, 2.0, 10.0])
    assert s == {"mean_ms": 4.0, "median_ms": 2.5, "min_ms": 1.0}


def test_clock_parser():
    text = (
        "index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], "
        "clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, "
        "clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, "
        "clocks_event_reasons.sw_power_cap\n"
        "0, 2032 MHz, 2032 MHz, 700 W, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1900 MHz, 2032 MHz, 1090 W, 0x4, Not Active, Not Active, Not Active, Active\n"
        "0, 2000 MHz, 2032 MHz, 900 W, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clock_csv(text)
    assert c["sm_mhz"] == 2000.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.parse_clock_csv("") is None


def test_workload_resolution():
    assert bench.resolve_workload(None).name == bench.DEFAULT_WORKLOAD
    assert bench.resolve_workload("5").index == 5
    assert bench.resolve_workload("paged_bf16_b128_h128_lvar").index == 4
