"""Benchmark of one MLA absorbed-decode step on B300.

One step = mla_absorb_q -> mla_decode_fwd -> mla_combine -> mla_out_proj over
one of the five seeded synthetic workloads (default: the DeepSeek-V3-shaped
one, B=64 sequences, h=128 heads, L=8192 cached tokens each, bf16, d_c=512,
d_r=64), inputs resident in HBM.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5 | NAME] [--parts P]

Timing: the clock sampler starts first, then untimed steps run for
--settle-s seconds (so that the SM and memory clocks sit at their loaded
state), then W warm-up steps, then exactly K timed steps with no idle gap
in between.  CUDA events bracket every decode launch; the line reports the
mean, median and minimum of those per-launch times next to the whole-step
throughput.

The reference arm (--impl reference) times the float64 CPU oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "v3_bf16_b64_h128_l8192"
METRIC = "MLA decode: latent-cache GB/s & TFLOP/s vs roofline (h=128, B=64, L=8k)"
UNIT = "GB/s"
PEAK_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 1024 * 1024


# ----------------------------------------------------------------------------
# host-side helpers (covered by CPU tests with gloo ranks)
# ----------------------------------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the torchrun environment (1 process if absent)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed / the slowest rank's time."""
    return per_rank_units * world / max_seconds


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAK_FALLBACK), "fallback"


def roofline(alg_bytes: float, alg_flops: float, seconds: float, hbm_gbs: float,
             tc_tflops: float) -> dict:
    """Roofline of one kernel launch: the bound is the slower of moving its
    algorithmic bytes at the HBM peak and doing its flops at the tensor peak;
    frac = that bound's time / the measured time (= achieved / peak of the bound)."""
    t_mem = alg_bytes / (hbm_gbs * 1e9)
    t_tc = alg_flops / (tc_tflops * 1e12)
    if t_mem >= t_tc:
        achieved, peak, unit, bound = alg_bytes / seconds / 1e9, hbm_gbs, "GB/s", "hbm"
    else:
        achieved, peak, unit, bound = alg_flops / seconds / 1e12, tc_tflops, "TFLOP/s", "tensor"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "t_mem_us": t_mem * 1e6, "t_tensor_us": t_tc * 1e6}


def step_stats(ms: list[float]) -> dict:
    """Mean, median and minimum of per-launch times (milliseconds)."""
    return {"mean_ms": statistics.fmean(ms), "median_ms": statistics.median(ms),
            "min_ms": min(ms)}


def parse_clock_csv(text: str) -> dict | None:
    """Median SM clock, max clock and the throttle reasons seen, from the
    nvidia-smi query recorded during the timed region."""
    rows = [r.strip() for r in text.strip().splitlines() if r.strip()]
    if len(rows) < 2:
        return None
    head = [h.strip() for h in rows[0].split(",")]
    data = [[c.strip() for c in r.split(",")] for r in rows[1:] if not r.startswith("index")]

    def col(name):
        for i, h in enumerate(head):
            if h.startswith(name):
                return i
        return None

    i_sm, i_max = col("clocks.current.sm"), col("clocks.max.sm")
    if i_sm is None:
        i_sm = col("clocks.sm")
    sm = [float(r[i_sm].split()[0]) for r in data if i_sm is not None and len(r) > i_sm
          and r[i_sm].split()[0].replace(".", "").isdigit()]
    mx = [float(r[i_max].split()[0]) for r in data if i_max is not None and len(r) > i_max
          and r[i_max].split()[0].replace(".", "").isdigit()]
    reasons = set()
    for name in ("clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                 "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"):
        i = col(name)
        if i is not None and any(len(r) > i and r[i] == "Active" for r in data):
            reasons.add(name.split(".")[-1])
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(sm)}


class ClockSampler:
    """nvidia-smi sampling of the SM clock and throttle reasons while running
    (reads only; nothing is set)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def result(self) -> dict | None:
        try:
            with open(self.path) as f:
                return parse_clock_csv(f.read())
        except OSError:
            return None
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass


def profile_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"decode_tc_{workload}.md")


def read_profile_traffic(workload: str, kernel_sha: str) -> float | None:
    """DRAM bytes per launch of the decode kernel on this workload from the
    committed ncu summary, if it was taken on this exact kernel source."""
    try:
        text = open(profile_path(workload)).read()
    except OSError:
        return None
    sha = traffic = None
    for line in text.splitlines():
        if line.startswith("kernel_source_sha256:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if sha == kernel_sha else None


def kernel_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_72_b300", "csrc")
    for name in ("decode_tc.cu", "common.cuh", "tc_ptx.cuh"):
        p = os.path.join(csrc, name)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def resolve_workload(arg):
    import mla_inputs as mi
    if arg is None:
        return mi.workload(DEFAULT_WORKLOAD)
    if isinstance(arg, str) and arg.isdigit():
        arg = int(arg)
    return mi.workload(arg)


def bench_config(w, num_parts, l2_note, q_len=1) -> dict:
    return {"workload": w.name, "B": w.B, "h": w.h, "L": w.L, "q_len": q_len,
            "L_range": list(w.L_range) if w.L_range else None, "d_c": w.d_c, "d_r": w.d_r,
            "d_nope": w.d_nope, "d_v": w.d_v, "cache_dtype": w.latent_dtype,
            "layout": w.layout, "block_size": w.block_size, "num_parts": num_parts,
            "l2": l2_note,
            "parallelism": "independent replica per GPU (batch-parallel, no collective)"}


# ----------------------------------------------------------------------------
# CPU baseline (the float64 oracle)
# ----------------------------------------------------------------------------

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(w, budget_s: float, start: int = 0):
    """Time the oracle (the non-absorbed definition) on windows of heads of
    whole sequences until about budget_s has elapsed.  Returns (attributed
    cache bytes, seconds, description, cores); each window is charged its
    share H/h of the sequence's cache bytes."""
    import oracle as O
    inp = O.workload_inputs_f64(w)
    per_tok = O.mla_cache_bytes_per_token(w.latent_dtype, w.dtype, w.d_c, w.d_r, w.block_size)
    seq_cache = {}

    def seq(b):
        if b not in seq_cache:
            seq_cache.clear()
            seq_cache[b] = O.sequence_view(w, b, int(inp["lens"][b]))
        return seq_cache[b]

    def run(b, heads):
        s = seq(b)
        t0 = time.perf_counter()
        O.decode_reference(inp["q_nope"][[b]], inp["q_rope"][[b]], inp["q_pos"][[b]],
                           inp["w_uk"], inp["w_uv"], [s], heads=heads)
        return time.perf_counter() - t0

    # heads per window: the whole head set unless one head already takes a
    # sizeable share of the budget
    t1 = run(start % w.B, [0])
    H = int(max(1, min(w.h, (budget_s / 4) // max(t1, 1e-6))))
    total_t, total_bytes, windows = 0.0, 0.0, 0
    i = 0
    while total_t < budget_s and windows < 4 * w.B:
        b = (start + i) % w.B
        h0 = (i * H) % w.h
        heads = [(h0 + k) % w.h for k in range(H)]
        total_t += run(b, heads)
        total_bytes += int(inp["lens"][b]) * per_tok * H / w.h
        windows += 1
        i += 1
    desc = (f"{windows} window(s) of {H} of {w.h} heads of whole sequences of the workload, "
            f"cache bytes attributed pro rata (H/h of each sequence's cache), float64 numpy, "
            f"{total_t:.1f} s")
    return total_bytes, total_t, desc, blas_threads()


def run_reference(args) -> None:
    """--impl reference: the float64 oracle on the host cores, K timed steps of a
    bounded sample each (a window of heads of one sequence per step)."""
    import oracle as O
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = resolve_workload(args.workload)
    inp = O.workload_inputs_f64(w)
    per_tok = O.mla_cache_bytes_per_token(w.latent_dtype, w.dtype, w.d_c, w.d_r, w.block_size)
    seq_cache = {}

    def seq(b):
        if b not in seq_cache:
            seq_cache.clear()
            seq_cache[b] = O.sequence_view(w, b, int(inp["lens"][b]))
        return seq_cache[b]

    def one(b, heads):
        s = seq(b)
        t0 = time.perf_counter()
        O.decode_reference(inp["q_nope"][[b]], inp["q_rope"][[b]], inp["q_pos"][[b]],
                           inp["w_uk"], inp["w_uv"], [s], heads=heads)
        return time.perf_counter() - t0

    # calibrate: seconds per head, then heads per step so that the run takes ~2 minutes
    t1 = one(0, [0])
    budget = float(os.environ.get("MLA_REFERENCE_BUDGET_S", "120"))
    per_step = budget / max(1, args.steps + args.warmup)
    H = int(max(1, min(w.h, per_step // max(t1, 1e-6))))
    total_t, total_bytes = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        b = i % w.B
        h0 = (i * H) % w.h
        heads = [(h0 + k) % w.h for k in range(H)]
        dt = one(b, heads)
        if i >= args.warmup:
            total_t += dt
            total_bytes += int(inp["lens"][b]) * per_tok * H / w.h
    value = total_bytes / total_t / 1e9
    sample = (f"{H} of {w.h} heads of one sequence per step, cache bytes attributed "
              f"pro rata (H/h of the sequence's cache)")
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(w, None, "host run: no GPU cache involved"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    from mla_latent_kv_72_b300 import binding as C
    from mla_latent_kv_72_b300 import build as mbuild
    from mla_latent_kv_72_b300.workload import DeviceWorkload

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        mbuild.build()
    barrier()
    C.lib()
    w = resolve_workload(args.workload)
    if args.batch is not None:
        import mla_inputs as mi
        w = mi.scaled(w, B=args.batch)
    parts = args.parts
    if parts is None and args.q_len > 1:
        # one CTA pair per part and per 128 query rows: keep one wave of pairs
        groups = (args.q_len * w.h + 127) // 128
        parts = max(1, C.default_num_parts(local) // groups)
    dw = DeviceWorkload(w, device=f"cuda:{local}", num_parts=parts, q_len=args.q_len)
    stream = torch.cuda.current_stream()

    # inputs of one step smaller than L2 are flushed from it between timed
    # steps (outside the per-step events); larger ones stream through it
    per_step_in = dw.cache_bytes()
    flush = per_step_in < 2 * L2_BYTES
    scrub = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dw.device) \
        if flush else None
    l2_note = (f"L2 flushed between timed steps by writing {2 * L2_BYTES >> 20} MiB "
               f"(outside the per-step events)" if flush else
               f"inputs larger than L2 ({per_step_in / 1e6:.0f} MB of latent cache per step)")

    n_st = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_st)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # settle: untimed steps until the clocks sit at their loaded state
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < args.settle_s:
            for _ in range(8):
                dw.step()
            torch.cuda.synchronize()
        for _ in range(args.warmup):
            dw.step()
        torch.cuda.synchronize()
        if dw.check_status() != 0:
            raise RuntimeError(f"device status {dw.check_status()} after warm-up")
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        # events bracket the decode kernel every step; the step boundaries get
        # events only when a flush runs between steps (otherwise start..end
        # times the steps back to back, and fewer events mean fewer gaps)
        for i in range(n_st):
            if flush:
                scrub.fill_(float(i))
                ev[i][0].record(stream)
            dw.absorb()
            ev[i][1].record(stream)
            dw.attend()
            ev[i][2].record(stream)
            dw.tail()
            if flush:
                ev[i][3].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
    clocks = clk.result()
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if flush:
        step_ms = [e[0].elapsed_time(e[3]) for e in ev]
        total_s = sum(step_ms) / 1e3
    else:
        total_s = start.elapsed_time(end) / 1e3
        step_ms = [total_s * 1e3 / n_st]       # back to back: the mean only
    max_total = reduce_max(total_s)
    assert dw.check_status() == 0

    step_bytes = dw.step_bytes()
    step_flops = dw.step_flops()
    value = aggregate(step_bytes * n_st, world, max_total) / 1e9
    tflops = aggregate(step_flops * n_st, world, max_total) / 1e12

    # end to end through the C ABI: every step copies its inputs in from pinned
    # host memory and its output back.  Two sets of device inputs and outputs
    # let the copies of steps k+1 and k-1 run on their own streams (the copy
    # engines) while step k computes, as a decode loop would overlap them.
    h_qn = dw.q_nope.cpu().pin_memory()
    h_qr = dw.q_rope.cpu().pin_memory()
    h_pos = dw.q_pos.cpu().pin_memory()
    h_out = [torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory() for _ in range(2)]
    h2d = h_qn.numel() * h_qn.element_size() + h_qr.numel() * h_qr.element_size() + \
        h_pos.numel() * h_pos.element_size()
    d2h = h_out[0].numel() * h_out[0].element_size()
    e2e_steps = max(3, min(n_st, 200))
    d_in = [(dw.q_nope, dw.q_rope, dw.q_pos),
            tuple(torch.empty_like(t) for t in (dw.q_nope, dw.q_rope, dw.q_pos))]
    d_out = [dw.out, torch.empty_like(dw.out)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of set i landed
    ev_used = [torch.cuda.Event() for _ in range(2)]    # the step using set i finished
    ev_read = [torch.cuda.Event() for _ in range(2)]    # output of set i copied out

    def e2e_step(k):
        i = k % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[i])
            for dst, src in zip(d_in[i], (h_qn, h_qr, h_pos)):
                dst.copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_read[i])
        dw.q_nope, dw.q_rope, dw.q_pos = d_in[i]
        dw.out = d_out[i]
        dw.step(stream=stream)
        ev_used[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[i])
            h_out[i].copy_(d_out[i], non_blocking=True)
            ev_read[i].record(s_out)

    def e2e_join():
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    for k in range(3):
        e2e_step(k)
    e2e_join()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(e2e_steps):
        e2e_step(k)
    e2e_join()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3)
    e2e_value = aggregate(step_bytes * e2e_steps, world, e2e_s) / 1e9
    assert torch.equal(h_out[0], h_out[1])      # same inputs, same outputs
    dw.q_nope, dw.q_rope, dw.q_pos = d_in[0]
    dw.out = d_out[0]

    breakdown = kernel_breakdown(dw, stream, flush, scrub)
    append = time_append(dw, stream, n_st)
    hidden = time_hidden(dw, args.hidden) if args.hidden else None

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    hbm = float(peaks.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
    tc_burst = float(peaks.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"]))
    tc_sust = float(peaks.get("bf16_tflops_sustained", PEAK_FALLBACK["bf16_tflops_sustained"]))
    dec_bytes, dec_flops = dw.decode_bytes(), dw.decode_flops()
    dstat = step_stats(dec_ms)
    dec_s = dstat["mean_ms"] / 1e3
    roof = roofline(dec_bytes, dec_flops, dec_s, hbm, tc_burst)
    sha = kernel_source_sha()
    roof.update({
        "traffic": read_profile_traffic(w.name, sha),
        "kernel": "mla_decode_fwd", "kernel_source_sha256": sha,
        "peak_source": f"{peak_kind} MEASURED_PEAKS.json (hbm_gbs; bf16_tflops burst)",
        "alg_bytes": dec_bytes, "alg_flops": dec_flops,
        "decode_ms": dstat["mean_ms"], "decode_median_ms": dstat["median_ms"],
        "decode_min_ms": dstat["min_ms"],
        "frac_at_median": roofline(dec_bytes, dec_flops, dstat["median_ms"] / 1e3, hbm,
                                   tc_burst)["frac"],
        "hbm_frac": dec_bytes / dec_s / 1e9 / hbm,
        "tensor_frac_burst": dec_flops / dec_s / 1e12 / tc_burst,
        "tensor_frac_sustained": dec_flops / dec_s / 1e12 / tc_sust,
    })

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        nbytes, secs, desc, cores = oracle_sample(w, args.cpu_budget)
        cpu = {"value": nbytes / secs / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc}
    sstat = step_stats(step_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_st,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_total / n_st,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic", "config": bench_config(w, dw.num_parts, l2_note, dw.q_len),
        "tflops": tflops, "steps_per_s": n_st / max_total,
        "step_ms": sstat,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": "pinned host buffers; inputs in and output out on two copy "
                          "streams, double-buffered, overlapping the neighbouring steps"},
        "kernels": breakdown,
        "append": append,
        "hidden": hidden,
        "gpu_launches": dw.launches_per_step() * n_st,
        "clocks": clocks,
        "settle_s": args.settle_s,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def time_append(dw, stream, steps: int) -> dict:
    """Per-launch time of mla_cache_append (one token per sequence), the
    cache write of each decode step: every call rewrites each sequence's last
    token (position L_b - 1) with its own data, so the cache is unchanged."""
    import numpy as np
    import torch

    import mla_inputs as mi
    from mla_latent_kv_72_b300 import binding as C
    from mla_latent_kv_72_b300.workload import storage_to_torch
    w = dw.w
    last = [mi.sequence_last_row(w, b, int(dw.lens_np[b])) for b in range(w.B)]
    c = np.stack([r[0] for r in last])
    kr = np.stack([r[1] for r in last])
    c_t = storage_to_torch(c, mi.latent_source_dtype(w), dw.device)
    kr_t = storage_to_torch(kr, w.dtype, dw.device)
    pos = torch.from_numpy((dw.lens_np - 1).astype(np.int32)).to(dw.device)
    def launch():
        C.mla_cache_append(c_t, kr_t, pos, dw.block_table, dw.kv, rope_theta=w.theta,
                           dev_status=dw.status)

    # the launches are replayed from a CUDA graph, so that the events time the
    # GPU work and not the host's launch overhead (a lone small kernel on an
    # idle GPU would otherwise wait for its own launch)
    per_graph = 50
    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            launch()
    torch.cuda.synchronize()
    n = max(3, min(steps // 10, 20))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    us = [a.elapsed_time(b) * 1e3 / per_graph for a, b in ev]
    per_tok = C.mla_cache_bytes_per_token(
        {"f32": 0, "bf16": 1, "fp8e4m3": 2}[w.latent_dtype], 0 if w.dtype == "f32" else 1,
        w.d_c, w.d_r, w.block_size)
    return {"kernel": "mla_cache_append", "tokens_per_launch": w.B,
            "mean_us": statistics.fmean(us), "median_us": statistics.median(us),
            "min_us": min(us), "written_bytes_per_launch": w.B * per_tok,
            "position": "each sequence's last token rewritten with its own data",
            "timing": f"CUDA events around graph replays of {per_graph} launches"}


def graph_time_us(fn, replays: int = 10, per_graph: int = 10) -> dict:
    """Per-call GPU time of fn from CUDA-graph replays (no host launch overhead)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 / per_graph for a, b in ev]
    return {"mean_us": statistics.fmean(us), "median_us": statistics.median(us), "min_us": min(us)}


def kernel_breakdown(dw, stream, flush: bool, scrub, steps: int = 50) -> dict:
    """Per-kernel device time of the step (after the timed region): events
    between the launches of each of `steps` further steps, so that every
    kernel sees the cache state it has inside a step (the weights of absorb
    and the projection come from HBM after the decode's stream has passed)."""
    import torch
    calls = [("mla_absorb_q", dw.absorb), ("mla_decode_fwd", dw.attend)]
    if dw.fused_tail:
        calls.append(("mla_combine_out_proj", dw.combine_project))
    else:
        calls += [("mla_combine", dw.combine), ("mla_out_proj", dw.project)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
          for _ in range(steps)]
    for i in range(steps):
        if flush:
            scrub.fill_(float(i))
        ev[i][0].record(stream)
        for k, (_, fn) in enumerate(calls):
            fn()
            ev[i][k + 1].record(stream)
    torch.cuda.synchronize()
    out = {}
    for k, (n, _) in enumerate(calls):
        us = [e[k].elapsed_time(e[k + 1]) * 1e3 for e in ev]
        out[n] = {"median_us": statistics.median(us), "min_us": min(us)}
    out["steps"] = steps
    return out


def time_hidden(dw, spec: str) -> dict:
    """The linear layers at the hidden-state boundary of the step (query
    compression x -> c_q -> q_nope, q_rope; output W_UV then W_O, or the
    merged W_O W_UV), per call, from CUDA-graph replays."""
    d_model, d_cq = (int(v) for v in spec.split(","))
    dw.enable_hidden(d_model, d_cq)
    w = dw.w
    res = {"d_model": d_model, "d_cq": d_cq}
    res["query_from_hidden"] = graph_time_us(dw.query_from_hidden)
    res["out_w_uv_then_w_o"] = graph_time_us(lambda: dw.hidden_out(False))
    dw.hidden_out(True)   # forms the merged matrix once (outside the timing)
    res["out_folded"] = graph_time_us(lambda: dw.hidden_out(True))
    el = 2
    res["weight_bytes"] = {
        "w_dq_w_uq_w_qr": el * d_cq * (d_model + w.h * (w.d_nope + w.d_r)),
        "w_uv_plus_w_o": el * w.h * w.d_v * (w.d_c + d_model),
        "w_fold": el * w.h * w.d_c * d_model}
    return res


def run_prefill(args) -> None:
    """--mode prefill: causal attention of whole prompts in the MHA form."""
    import torch

    import mla_inputs as mi
    from mla_latent_kv_72_b300 import build as mbuild
    from mla_latent_kv_72_b300.workload import DevicePrefill
    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    mbuild.build()
    w = resolve_workload(args.workload)
    w = mi.scaled(w, B=args.batch if args.batch is not None else 4)
    pf = DevicePrefill(w, device=f"cuda:{local}")
    for _ in range(args.warmup):
        pf.run()
    torch.cuda.synchronize()
    att = graph_time_us(pf.attend, replays=max(3, min(args.steps, 20)), per_graph=2)
    kv = graph_time_us(pf.keys_values, replays=5, per_graph=2)
    q = graph_time_us(pf.query, replays=5, per_graph=2)
    assert pf.dw.check_status() == 0
    peaks, peak_kind = load_peaks()
    tc = float(peaks.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"]))
    flops = pf.attention_flops()
    t = att["mean_us"] * 1e-6
    line = {"metric": "MLA prefill attention, MHA form (causal, d_qk=192, d_v=128): TFLOP/s",
            "value": flops / t / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": att["mean_us"] / 1e3,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "h": w.h, "L": w.L,
                       "tokens": pf.T, "mode": "prefill"},
            "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": tc,
                         "unit": "TFLOP/s", "frac": flops / t / 1e12 / tc,
                         "peak_source": f"{peak_kind} bf16_tflops (burst)",
                         "kernel": "mla_prefill_fwd", "alg_flops": flops},
            "attention": att, "keys_values_mla_linear": kv, "query": q}
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None,
                   help="workload index 1..5 or name (default: the V3-shaped workload, 3)")
    p.add_argument("--parts", type=int, default=None,
                   help="balanced parts of the block stream (default: half the SM count)")
    p.add_argument("--batch", type=int, default=None,
                   help="sequences of the workload (default: its own B; a smaller B makes a "
                        "profiling case of the same kernel)")
    p.add_argument("--q-len", type=int, default=1,
                   help="new tokens per sequence (multi-token decode; 1 = the one-token step)")
    p.add_argument("--settle-s", type=float, default=0.5,
                   help="seconds of untimed steps before the warm-up")
    p.add_argument("--mode", choices=["decode", "prefill"], default="decode")
    p.add_argument("--hidden", default=None,
                   help="D_MODEL,D_CQ: also time the linear layers at the hidden-state boundary")
    p.add_argument("--cpu-budget", type=float, default=15.0,
                   help="seconds of oracle work for the CPU baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.mode == "prefill":
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
