"""Benchmark of one MLA absorbed-decode step on B300.

One step = mla_absorb_q -> mla_decode_fwd -> mla_combine -> mla_out_proj over
the DeepSeek-V3-shaped workload (B=64 sequences, h=128 heads, L=8192 cached
tokens each, bf16, d_c=512, d_r=64), synthetic seeded inputs resident in HBM.
Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

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

WORKLOAD = "v3_bf16_b64_h128_l8192"
METRIC = "MLA decode: latent-cache GB/s & TFLOP/s vs roofline (h=128, B=64, L=8k)"
UNIT = "GB/s"
PEAK_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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
    """nvidia-smi sampling of the SM clock and throttle reasons while running."""

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
        time.sleep(0.3)
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


def read_profile_traffic(kernel_sha: str) -> float | None:
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    if it was taken on this exact kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_tc_v3_bf16_b64_h128_l8192.md")
    try:
        text = open(path).read()
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


# ----------------------------------------------------------------------------
# CPU baseline (the float64 oracle)
# ----------------------------------------------------------------------------

def oracle_sample(w, budget_s: float, start_b: int = 0):
    """Time the oracle on whole sequences (all heads) until about budget_s has
    elapsed; return (attributed cache bytes, seconds, sequences, cores)."""
    import numpy as np

    import mla_inputs as mi
    import oracle as O
    inp = O.workload_inputs_f64(w)
    per_tok = O.mla_cache_bytes_per_token(w.latent_dtype, w.dtype, w.d_c, w.d_r, w.block_size)
    total_t, total_bytes, nseq = 0.0, 0.0, 0
    b = start_b
    while total_t < budget_s and nseq < w.B:
        L = int(inp["lens"][b])
        seqs = [O.sequence_view(w, b, L)]
        t0 = time.perf_counter()
        O.decode_reference(inp["q_nope"][[b]], inp["q_rope"][[b]], inp["q_pos"][[b]],
                           inp["w_uk"], inp["w_uv"], seqs)
        total_t += time.perf_counter() - t0
        total_bytes += L * per_tok
        nseq += 1
        b = (b + 1) % w.B
    return total_bytes, total_t, nseq, blas_threads()


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args) -> None:
    """--impl reference: the float64 oracle on the host cores, K timed steps of a
    bounded sample each (a window of heads of one sequence per step)."""
    import numpy as np

    import mla_inputs as mi
    import oracle as O
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = mi.workload(WORKLOAD)
    inp = O.workload_inputs_f64(w)
    per_tok = O.mla_cache_bytes_per_token(w.latent_dtype, w.dtype, w.d_c, w.d_r, w.block_size)
    seq_cache = {}

    def seq(b):
        if b not in seq_cache:
            seq_cache.clear()
            seq_cache[b] = O.sequence_view(w, b, int(inp["lens"][b]))
        return seq_cache[b]

    def one(b, heads):
        t0 = time.perf_counter()
        O.decode_reference(inp["q_nope"][[b]], inp["q_rope"][[b]], inp["q_pos"][[b]],
                           inp["w_uk"], inp["w_uv"], [seq(b)], heads=heads)
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
    sample = (f"{H} of {w.h} heads of one sequence (L={w.L}) per step, cache bytes attributed "
              f"pro rata (H/h of the sequence's cache)")
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(w, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_config(w, num_parts) -> dict:
    return {"workload": w.name, "B": w.B, "h": w.h, "L": w.L, "d_c": w.d_c, "d_r": w.d_r,
            "d_nope": w.d_nope, "d_v": w.d_v, "cache_dtype": w.latent_dtype,
            "block_size": w.block_size, "num_parts": num_parts,
            "l2": "inputs larger than L2 (604 MB latent cache per step)",
            "parallelism": "independent replica per GPU (batch-parallel, no collective)"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    import mla_inputs as mi
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
    w = mi.workload(WORKLOAD)
    dw = DeviceWorkload(w, device=f"cuda:{local}", num_parts=args.parts)
    stream = torch.cuda.current_stream()

    # warm-up
    for _ in range(args.warmup):
        dw.step()
    torch.cuda.synchronize()
    if dw.check_status() != 0:
        raise RuntimeError(f"device status {dw.check_status()} after warm-up")

    # timed region: K steps, events around every decode launch for the roofline
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            dw.absorb()
            ev_s[i].record(stream)
            dw.attend()
            ev_e[i].record(stream)
            dw.combine()
            dw.project()
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
    clocks = clk.result()
    total_s = start.elapsed_time(end) / 1e3
    decode_s = sum(a.elapsed_time(b) for a, b in zip(ev_s, ev_e)) / 1e3 / args.steps
    max_total = reduce_max(total_s)
    assert dw.check_status() == 0

    step_bytes = dw.step_bytes()
    step_flops = dw.step_flops()
    value = aggregate(step_bytes * args.steps, world, max_total) / 1e9
    tflops = aggregate(step_flops * args.steps, world, max_total) / 1e12

    # end to end through the C ABI: pinned host inputs in, output back, every step
    h_qn = dw.q_nope.cpu().pin_memory()
    h_qr = dw.q_rope.cpu().pin_memory()
    h_pos = dw.q_pos.cpu().pin_memory()
    h_out = torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory()
    h2d = h_qn.numel() * h_qn.element_size() + h_qr.numel() * h_qr.element_size() + \
        h_pos.numel() * h_pos.element_size()
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step():
        dw.q_nope.copy_(h_qn, non_blocking=True)
        dw.q_rope.copy_(h_qr, non_blocking=True)
        dw.q_pos.copy_(h_pos, non_blocking=True)
        dw.step()
        h_out.copy_(dw.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3)
    e2e_value = aggregate(step_bytes * e2e_steps, world, e2e_s) / 1e9

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    hbm = float(peaks.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
    tc = float(peaks.get("bf16_tflops_sustained", PEAK_FALLBACK["bf16_tflops_sustained"]))
    dec_bytes = dw.cache_bytes() + w.B * w.h * (w.d_c + w.d_r) * 2 + dw.table_np.size * 4 + w.B * 4
    dec_flops = float(dw.lens_np.sum()) * w.h * 2 * (w.d_c + w.d_r + w.d_c)
    achieved = dec_bytes / decode_s / 1e9
    sha = kernel_source_sha()
    traffic = read_profile_traffic(sha)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        nbytes, secs, nseq, cores = oracle_sample(w, args.cpu_budget)
        cpu = {"value": nbytes / secs / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{nseq} whole sequence(s) of the workload (L={w.L}, all {w.h} heads), "
                         f"float64 numpy, {secs:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": bench_config(w, dw.num_parts),
        "tflops": tflops, "steps_per_s": args.steps / max_total,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": "mla_decode_fwd", "peak_source": f"{peak_kind} hbm_gbs",
                     "decode_ms": decode_s * 1e3,
                     "tensor_frac": dec_flops / decode_s / 1e12 / tc,
                     "tensor_peak_tflops": tc},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--parts", type=int, default=None,
                   help="balanced parts of the block stream (default: half the SM count)")
    p.add_argument("--cpu-budget", type=float, default=15.0,
                   help="seconds of oracle work for the CPU baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
