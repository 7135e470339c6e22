#!/usr/bin/env python
"""Benchmark of the Parallax attention layer (forward + backward) on B300.

One step = one pass of the whole layer: forward (pass 1, projection, pass 2)
and backward (dq, dk, dv, dP) over one batch of the workload
``c4`` (causal, bf16, B=8, H=16, T=4096, d=64; q, k, v, dO ~ N(0,1),
P_h ~ N(0, (0.1/sqrt(d))^2), seed 3), inputs resident in HBM.

Metric: algorithmic TFLOP/s of the step (28 d flops per causal pair: 8 d
forward, 20 d backward) and its fraction of the measured bf16 tensor peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs its own independent set of heads (weak scaling, no collective on the
data path) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import plx_synth  # noqa: E402

METRIC = "Parallax attn fwd/bwd TFLOP/s & % of B300 bf16 tensor peak, T=4096"
UNIT = "TFLOP/s"
L2_BYTES = 126 * 1024 * 1024

# Algorithmic flops per causal pair, per kernel role (each MMA-shaped product
# counted once: S, mu_k | G, o | S, E, R | G, Y, dV, dK (3 terms), dQ).
FWD_FLOPS_PER_PAIR_D = 8
BWD_FLOPS_PER_PAIR_D = 20
# MMA flops the forward executes per causal pair: pass 1 S and P~K (4d),
# pass 2 S, G and W V (6d); S is computed twice.
FWD_EXEC_FLOPS_PER_PAIR_D = 10
KERNEL_FLOPS_PER_PAIR_D = {
    "tc_pass1": 4, "simt_pass1": 4,
    "tc_pass2": 4, "simt_pass2": 4,
    "tc_bwd_b1": 6, "simt_bwd_b1": 6,
    "tc_bwd_b3": 14, "simt_bwd_b3": 14,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "sm_max_mhz": p.get("sm_max_mhz", 2032.0), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "sm_max_mhz": 2032.0, "source": "fallback"}


def measured_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None
    when there is none or the kernel's source changed since it was taken.  Each
    entry names the source file and the two lines that bound the kernel's text;
    the hash covers that text only, so editing another kernel of the same file
    does not void it."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic_c4.json")
    try:
        with open(path) as f:
            doc = json.load(f)
        k = doc["kernels"][kernel]
        with open(os.path.join(ROOT, k["source"])) as f:
            src = f.read()
        i0 = src.index(k["begin"])
        i1 = src.index(k["end"], i0)
        if hashlib.sha256(src[i0:i1].encode()).hexdigest() != k["sha256"]:
            return None
        return k["read"] + k["write"]
    except (OSError, KeyError, ValueError):
        return None


def fp32_simt_peak_tflops(sm_mhz: float) -> float:
    # 148 SMs x 128 FP32 lanes x 2 flops (FFMA) per clock
    return 148 * 128 * 2 * sm_mhz * 1e6 / 1e12


# ------------------------------------------------------------------ dist
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws an independent set of heads (weak scaling)."""
    return base + 7919 * rank


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="plx_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
               "-f", self.path]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for r in csv.reader(io.StringIO(f.read())):
                    if len(r) >= 9:
                        rows.append([x.strip() for x in r])
        finally:
            os.unlink(self.path)
        return summarize_clocks(rows)


def summarize_clocks(rows) -> dict:
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
            power.append(float(r[3]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    # samples under load: the upper half of the observed clocks/power
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
            "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


def gpu_query_id(torch, dev) -> str | None:
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", 0)
        devid = getattr(props, "pci_device_id", 0)
        if bus is not None:
            return f"{dom:08X}:{bus:02X}:{devid:02X}.0"
    except Exception:
        pass
    return None


# ----------------------------------------------------------- CPU baseline
def oracle_sample(inp: dict, nheads: int, rows: int, threads: int) -> tuple[float, int]:
    """Time the oracle's forward + backward on `nheads` heads (batch 0) over
    the first `rows` queries (and keys).  Returns (seconds, causal pairs)."""
    import oracle
    d = inp["d"]
    sl = (slice(0, 1), slice(0, nheads), slice(0, rows))
    q = plx_synth.widen(inp["q"][sl])
    k = plx_synth.widen(inp["k"][sl])
    v = plx_synth.widen(inp["v"][sl])
    do = plx_synth.widen(inp["dout"][sl])
    P = inp["P"][:nheads].astype(np.float64)
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(q, k, v, P, nthreads=threads)
    oracle.backward(q, k, v, P, do, nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, plx_synth.causal_pairs(1, nheads, rows)


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def calibrate_rows(inp, nheads, threads, target_s, T) -> int:
    """Largest row count (multiple of 64, <= T) whose sample takes ~target_s."""
    r0 = min(T, 512)
    dt, _ = oracle_sample(inp, nheads, r0, threads)
    if dt <= 0:
        return T
    scale = math.sqrt(target_s / dt)
    rows = int(min(T, max(64, r0 * scale)) // 64 * 64)
    return max(64, rows)


# ----------------------------------------------------------------- arms
def run_reference(args, world, rank):
    """The oracle (fp64 C loops) timed on this host's cores: the reference arm."""
    if rank != 0:
        return
    w = plx_synth.WORKLOADS[args.workload]
    inp = plx_synth.generate_workload(args.workload, B=1, H=w.H, backward=True)
    threads = cpu_threads()
    nheads = min(w.H, threads)
    budget = max(10.0, 150.0 / max(1, args.steps + args.warmup))
    rows = calibrate_rows(inp, nheads, threads, budget, w.T)
    for _ in range(args.warmup):
        oracle_sample(inp, nheads, rows, threads)
    tot_s, tot_pairs = 0.0, 0
    for _ in range(args.steps):
        dt, pairs = oracle_sample(inp, nheads, rows, threads)
        tot_s += dt
        tot_pairs += pairs
    flops = tot_pairs * (FWD_FLOPS_PER_PAIR_D + BWD_FLOPS_PER_PAIR_D) * w.d
    value = flops / tot_s / 1e12
    sample = (f"{nheads} heads x first {rows} queries/keys of one batch, fwd+bwd, per step "
              f"(full step: {w.B * w.H} heads x {w.T})")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_s / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "oracle"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, path):
    return {"workload": w.describe, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "path": path,
            "pairs_per_step": plx_synth.causal_pairs(w.B, w.H, w.T),
            "algorithmic_flops_per_pair": f"{FWD_FLOPS_PER_PAIR_D}d fwd + {BWD_FLOPS_PER_PAIR_D}d bwd",
            "l2": "inputs larger than L2 (q,k,v,dO: 4 x {:.0f} MB bf16 > 126 MB); no flush".format(
                w.B * w.H * w.T * w.d * 2 / 1e6)}


def run_ours(args, world, rank):
    import torch
    import parallax_local_linear_fwd_b300 as plx

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist_init("nccl")
    w = plx_synth.WORKLOADS[args.workload]
    if args.shard == "batch":
        # one problem split by batch: every rank draws the same inputs and
        # keeps its slice; dP_h is summed across ranks inside the step
        from parallax_local_linear_fwd_b300.shard import shard_range
        inp = plx_synth.generate_workload(args.workload, backward=True)
        lo, hi = shard_range(w.B, rank, world)
        if hi <= lo:
            raise SystemExit(f"--shard batch needs at least one batch per rank (B={w.B}, ranks={world})")
        inp = {n: (x[lo:hi] if n in ("q", "k", "v", "dout") else x) for n, x in inp.items()}
        B = hi - lo
    else:
        inp = plx_synth.generate_workload(args.workload, seed=rank_seed(w.seed, rank), backward=True)
        B = w.B
    H, T, d = w.H, w.T, w.d

    def host(x):
        if x.dtype == np.uint16:
            t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(x)
        return t.pin_memory()

    h_in = {k: host(inp[k]) for k in ("q", "k", "v", "P", "dout")}
    d_in = {k: t.to(dev) for k, t in h_in.items()}
    q, k, v, P, do = (d_in[x] for x in ("q", "k", "v", "P", "dout"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    mu = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dP = torch.empty_like(P)
    dtc = plx.PLX_BF16 if q.dtype == torch.bfloat16 else plx.PLX_FP32
    fws = torch.empty(max(256, plx.parallax_fwd_workspace_bytes(B, H, T, d, dtc)), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(256, plx.parallax_bwd_workspace_bytes(B, H, T, d, dtc)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    path = "tc" if _tc_ws(plx, B, H, T, d, dtc) > 0 else "simt"

    sws = torch.empty(max(256, plx.parallax_fwd_bwd_workspace_bytes(B, H, T, d, dtc)), dtype=torch.uint8, device=dev)

    def step():
        # one training step through the fused entry point (one workspace, the
        # backward reusing the forward's f16 operand copies)
        plx.parallax_fwd_bwd(q, k, v, P, do, out, lse, mu, dq, dk, dv, dP, workspace=sws, stream=stream)
        if args.shard == "batch" and world > 1:
            from parallax_local_linear_fwd_b300.shard import allreduce_dP
            allreduce_dP(dP)

    for _ in range(args.warmup):
        step()
    code, detail = plx.parallax_last_device_error(stream)
    if code != plx.PLX_OK:
        raise RuntimeError(f"device watchdog: {plx.parallax_strerror(code)} detail={detail:#x}")

    clocks = ClockSampler(gpu_query_id(torch, dev))
    clocks.start()
    time.sleep(0.3)
    plx.parallax_timing_reset()
    plx.parallax_timing_enable(True)
    n0 = plx.parallax_launch_count()
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    launches = plx.parallax_launch_count() - n0
    plx.parallax_timing_enable(False)
    kt = plx.kernel_times()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    code, detail = plx.parallax_last_device_error(stream)
    if code != plx.PLX_OK:
        raise RuntimeError(f"device watchdog: {plx.parallax_strerror(code)} detail={detail:#x}")

    pairs = plx_synth.causal_pairs(B, H, T)
    flops_step = pairs * (FWD_FLOPS_PER_PAIR_D + BWD_FLOPS_PER_PAIR_D) * d
    # the whole job's work per step: N independent problems (head replicas),
    # or one problem split by batch
    job_pairs = plx_synth.causal_pairs(w.B, H, T) if args.shard == "batch" else world * pairs
    job_flops_step = job_pairs * (FWD_FLOPS_PER_PAIR_D + BWD_FLOPS_PER_PAIR_D) * d
    value = job_flops_step * args.steps / (ms / 1e3) / 1e12
    peaks = load_peaks()

    # dominant kernel and its live roofline
    kernels = {}
    total_k_ms = sum(v_[0] for v_ in kt.values()) or 1.0
    for name, (tms, cnt) in kt.items():
        kernels[name] = {"launches": cnt, "avg_ms": tms / cnt, "share": tms / total_k_ms}
    dom = max(kt, key=lambda n: kt[n][0]) if kt else None
    roofline = None
    if dom is not None:
        avg_s = kt[dom][0] / kt[dom][1] / 1e3
        fpp = KERNEL_FLOPS_PER_PAIR_D.get(dom)
        if fpp is not None:
            achieved = pairs * fpp * d / avg_s / 1e12
            if dom.startswith("tc_"):
                # the timed region lasts well under a second: the burst peak
                # (a kernel timed alone), not the seconds-long sustained one
                peak, bound = peaks["bf16_tflops"], "tensor"
                peak_note = f"bf16 dense, {peaks['source']} burst (timed region under a second)"
            else:
                peak, bound = fp32_simt_peak_tflops(peaks["sm_max_mhz"]), "alu"
                peak_note = "fp32 FFMA: 148 SMs x 128 lanes x 2 x max SM clock"
            roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "traffic": measured_traffic(dom), "peak_source": peak_note,
                        "flops_per_launch": pairs * fpp * d}
    # whole-step fraction of the tensor peak
    pct_peak = flops_step * args.steps / (ms / 1e3) / 1e12 / peaks["bf16_tflops"]

    # forward / backward split (timed separately, same inputs)
    fwd_ms, bwd_ms = split_fwd_bwd(torch, plx, q, k, v, P, out, lse, mu, do, dq, dk, dv, dP, fws, bws, stream,
                                   max(3, args.steps // 2))

    # end to end through the public API with host buffers
    e2e = run_e2e(torch, plx, h_in, dev, stream, args, B, H, T, d, world, job_flops_step,
                  allreduce=args.shard == "batch" and world > 1)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "strong" if args.shard == "batch" else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_config(w, path),
                   "parallelism": (f"batch-shard x{world} (dP all-reduce)" if args.shard == "batch"
                                   else f"independent head sets x{world}")},
        "pct_of_bf16_peak": pct_peak,
        "tokens_per_s": (w.B if args.shard == "batch" else world * B) * T * args.steps / (ms / 1e3),
        "fwd": {"ms": fwd_ms, "tflops": pairs * FWD_FLOPS_PER_PAIR_D * d / (fwd_ms / 1e3) / 1e12},
        "bwd": {"ms": bwd_ms, "tflops": pairs * BWD_FLOPS_PER_PAIR_D * d / (bwd_ms / 1e3) / 1e12},
        "gpu_launches": launches,
        "kernels": kernels,
        "roofline": roofline,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_fwd_c3:
        line["decode"] = decode_workload(torch, plx, k, v, P, stream)
        if k.dtype == torch.bfloat16:
            line["decode_probe"] = decode_workload(torch, plx, k, v, P, stream, probe=True)
    if rank == 0 and world == 1 and path == "tc" and not args.no_fwd_c3:
        line["fwd_c3"] = forward_workload(torch, plx, "c3", dev, stream)
        line["fwd_probe_c3"] = probe_workload(torch, plx, "c3", dev, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_threads()
        nheads = min(H, threads)
        rows = calibrate_rows(inp, nheads, threads, 15.0, T)
        dt, sp = oracle_sample(inp, nheads, rows, threads)
        line["cpu_baseline"] = {"value": sp * (FWD_FLOPS_PER_PAIR_D + BWD_FLOPS_PER_PAIR_D) * d / dt / 1e12,
                                "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{nheads} heads x first {rows} queries/keys, fwd+bwd, fp64"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _tc_ws(plx, B, H, T, d, dtc):
    prev = plx.parallax_set_path(plx.PLX_PATH_TC)
    try:
        return plx.parallax_fwd_workspace_bytes(B, H, T, d, dtc) or -1
    finally:
        plx.parallax_set_path(prev)


def forward_workload(torch, plx, name, dev, stream, iters=10, warmup=3):
    """Forward-only throughput of another workload (c3: B4 H16 T4096 d128, the
    shape the forward target is stated on), inputs resident in HBM, timed with
    CUDA events on the launching stream; per-kernel shares from the library's
    event timing."""
    w = plx_synth.WORKLOADS[name]
    inp = plx_synth.generate_workload(name)
    B, H, T, d = w.B, w.H, w.T, w.d

    def dev_t(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    q, k, v, P = (dev_t(inp[x]) for x in ("q", "k", "v", "P"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    mu = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    dtc = plx.PLX_BF16
    fws = torch.empty(max(256, plx.parallax_fwd_workspace_bytes(B, H, T, d, dtc)), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        plx.parallax_fwd_ws(q, k, v, P, out, lse, mu, fws, stream=stream)
    # the forward as a caller runs it (no per-kernel events between its
    # launches), then the same loop again with the library's per-kernel events
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        plx.parallax_fwd_ws(q, k, v, P, out, lse, mu, fws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / iters
    plx.kernel_times()
    plx.parallax_timing_reset()
    plx.parallax_timing_enable(True)
    for _ in range(iters):
        plx.parallax_fwd_ws(q, k, v, P, out, lse, mu, fws, stream=stream)
    torch.cuda.synchronize(dev)
    plx.parallax_timing_enable(False)
    kt = plx.kernel_times()
    pairs = plx_synth.causal_pairs(B, H, T)
    peaks = load_peaks()
    alg = pairs * FWD_FLOPS_PER_PAIR_D * d / (ms / 1e3) / 1e12
    exe = pairs * FWD_EXEC_FLOPS_PER_PAIR_D * d / (ms / 1e3) / 1e12
    res = {"workload": w.describe, "ms": ms, "tflops_algorithmic": alg, "tflops_executed_mma": exe,
           "frac_of_bf16_peak_algorithmic": alg / peaks["bf16_tflops"],
           "frac_of_bf16_peak_executed": exe / peaks["bf16_tflops"], "peak": peaks["bf16_tflops"],
           "peak_source": f"bf16 dense, {peaks['source']} burst", "kernels": {},
           "timing": "ms: the forward alone, CUDA events around the loop; kernels: a second loop with "
                     "the library's per-kernel events"}
    for kname, (tms, cnt) in kt.items():
        avg = tms / cnt
        entry = {"avg_ms": avg}
        fpp = KERNEL_FLOPS_PER_PAIR_D.get(kname)
        if fpp is not None:
            entry["tflops_algorithmic"] = pairs * fpp * d / (avg / 1e3) / 1e12
        res["kernels"][kname] = entry
    del q, k, v, P, out, lse, mu, fws
    torch.cuda.empty_cache()
    return res


def decode_workload(torch, plx, k, v, P, stream, iters=20, warmup=3, probe=False):
    """Decode step over the step's own keys and values as a KV cache (one new
    query per head, every sequence at full length).  HBM-bound: the roofline
    is the measured copy bandwidth; the algorithmic bytes are the cache (K and
    V read once each).  probe=True times the given-probe form
    (parallax_decode_probe, a probe rho per head) instead of the projector's."""
    B, H, L, d = (int(x) for x in k.shape)
    gen = torch.Generator(device="cpu").manual_seed(17)
    q = torch.randn((B, H, d), generator=gen).to(k.dtype).to(k.device)
    rho = (0.3 * torch.randn((B, H, d), generator=gen)).to(k.dtype).to(k.device)
    out = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=k.device)
    dtc = plx.PLX_BF16 if k.dtype == torch.bfloat16 else plx.PLX_FP32
    wsb = (plx.parallax_decode_probe_workspace_bytes if probe else plx.parallax_decode_workspace_bytes)(B, H, L, d, dtc)
    ws = torch.empty(max(256, wsb), dtype=torch.uint8, device=k.device)

    def call(st):
        if probe:
            plx.parallax_decode_probe(q, k, v, rho, out=out, lse=lse, workspace=ws, stream=st)
        else:
            plx.parallax_decode(q, k, v, P, out=out, lse=lse, workspace=ws, stream=st)
    for _ in range(warmup):
        call(stream)
    # timed without the library's per-kernel events: at this microsecond
    # scale their host work per launch would be measured too
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        call(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / iters
    # the same step captured once in a CUDA graph and replayed, as a serving
    # loop runs it: device time with no host work between the launches
    cs = torch.cuda.Stream(device=k.device)
    cs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        call(cs)
    for _ in range(warmup):
        graph.replay()
    # the cache (2 x 67 MB) barely exceeds L2 (126 MB): every timed replay
    # starts after an untimed write of 256 MB, so K and V come from HBM.  A
    # read of another 256 MB follows the write, so the L2 holds clean lines
    # when the replay starts: without it the replay would also pay for
    # writing the flush buffer's ~126 MB of dirty lines back to HBM, a cost
    # a serving loop (whose step writes a few KB) does not have.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=k.device)
    clean = torch.zeros(32 << 20, dtype=torch.int64, device=k.device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    torch.cuda.synchronize()
    with torch.cuda.stream(cs):
        for a_, b_ in evs:
            flush.fill_(1)
            clean.sum()
            a_.record(cs)
            graph.replay()
            b_.record(cs)
    torch.cuda.synchronize()
    ms = sum(a_.elapsed_time(b_) for a_, b_ in evs) / iters
    del graph, flush, clean
    # a third loop with the library's events gives the per-kernel split
    plx.kernel_times()
    plx.parallax_timing_reset()
    plx.parallax_timing_enable(True)
    for _ in range(iters):
        call(stream)
    torch.cuda.synchronize()
    plx.parallax_timing_enable(False)
    kt = plx.kernel_times()
    cache_bytes = 2 * k.numel() * k.element_size()
    peaks = load_peaks()
    gbs = cache_bytes / (ms / 1e3) / 1e9
    form = "given probe rho per head" if probe else "probe formed by the projector P_h"
    return {"workload": f"decode, {str(k.dtype).replace('torch.', '')}, B{B} H{H} cache {L} d{d}, "
                        f"one new query per head, {form}", "us": ms * 1e3, "timing": "CUDA-graph replay of the call, L2 flushed before each",
            "l2": "256 MB written, then another 256 MB read, before each timed replay",
            "us_eager": ms_eager * 1e3, "tokens_per_s": B / (ms / 1e3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": cache_bytes,
                         "peak_source": f"{peaks['source']} copy bandwidth"},
            "kernels": {n: {"avg_us": 1e3 * t / c} for n, (t, c) in kt.items()}}


def probe_workload(torch, plx, name, dev, stream, iters=10, warmup=3):
    """One-pass given-probe forward on a workload's shape (rho drawn like the
    projector-formed probe's scale), inputs resident in HBM."""
    w = plx_synth.WORKLOADS[name]
    B, H, T, d = w.B, w.H, w.T, w.d
    gen = torch.Generator(device="cpu").manual_seed(23)
    mk = lambda s: (s * torch.randn((B, H, T, d), generator=gen)).to(torch.bfloat16).to(dev)  # noqa: E731
    q, k, v = mk(1.0), mk(1.0), mk(1.0)
    rho = mk(0.1 / math.sqrt(d))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, plx.parallax_fwd_probe_workspace_bytes(B, H, T, d, plx.PLX_BF16)), dtype=torch.uint8,
                     device=dev)
    for _ in range(warmup):
        plx.parallax_fwd_probe(q, k, v, rho, out=out, lse=lse, workspace=ws, stream=stream)
    plx.kernel_times()
    plx.parallax_timing_reset()
    plx.parallax_timing_enable(True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        plx.parallax_fwd_probe(q, k, v, rho, out=out, lse=lse, workspace=ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    plx.parallax_timing_enable(False)
    kt = plx.kernel_times()
    ms = e0.elapsed_time(e1) / iters
    pairs = plx_synth.causal_pairs(B, H, T)
    peaks = load_peaks()
    tf = pairs * 8 * d / (ms / 1e3) / 1e12  # S, R, O1, O2: 8 d flops per causal pair
    res = {"workload": f"one-pass given-probe forward, bf16, B{B} H{H} T{T} d{d}", "ms": ms, "tflops": tf,
           "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "peak_source": f"bf16 dense, {peaks['source']} burst",
           "kernels": {n: {"avg_ms": t / c} for n, (t, c) in kt.items()}}
    if "tc_probe" in kt:
        t_, c_ = kt["tc_probe"]
        res["kernels"]["tc_probe"]["tflops"] = pairs * 8 * d / (t_ / c_ / 1e3) / 1e12
    del q, k, v, rho, out, lse, ws
    torch.cuda.empty_cache()
    return res


def split_fwd_bwd(torch, plx, q, k, v, P, out, lse, mu, do, dq, dk, dv, dP, fws, bws, stream, n):
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for _ in range(n):
        plx.parallax_fwd_ws(q, k, v, P, out, lse, mu, fws, stream=stream)
    ev[1].record(stream)
    for _ in range(n):
        plx.parallax_bwd(q, k, v, P, lse, mu, do, dq, dk, dv, dP, workspace=bws, stream=stream)
    ev[2].record(stream)
    torch.cuda.synchronize()
    return ev[0].elapsed_time(ev[1]) / n, ev[1].elapsed_time(ev[2]) / n


def run_e2e(torch, plx, h_in, dev, stream, args, B, H, T, d, world, job_flops_step, allreduce=False):
    """Same step through the public host-buffer entry point, parallax_step_host:
    from pinned host inputs to pinned host outputs, with the H2D copies, the
    forward + backward and the D2H copies (overlapped by head groups) all
    inside the timed region."""
    h_out = {n: torch.empty(s, dtype=dt).pin_memory() for n, s, dt in (
        ("out", (B, H, T, d), h_in["q"].dtype), ("dq", (B, H, T, d), h_in["q"].dtype),
        ("dk", (B, H, T, d), h_in["q"].dtype), ("dv", (B, H, T, d), h_in["q"].dtype),
        ("dP", (H, d, d), torch.float32))}
    dP_dev = torch.empty(h_out["dP"].shape, dtype=torch.float32, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    chunks = min(H, 8)

    def step():
        plx.parallax_step_host(h_in["q"], h_in["k"], h_in["v"], h_in["P"], h_in["dout"], out=h_out["out"],
                               dq=h_out["dq"], dk=h_out["dk"], dv=h_out["dv"], dP=h_out["dP"], chunks=chunks,
                               stream=stream)
        if allreduce:
            # the batch-shard exchange: the host dP of every rank summed
            import torch.distributed as dist
            stream.synchronize()
            dP_dev.copy_(h_out["dP"])
            dist.all_reduce(dP_dev)
            h_out["dP"].copy_(dP_dev)

    n = max(3, args.steps // 2)
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    return {"value": job_flops_step * n / (ms / 1e3) / 1e12, "unit": UNIT, "steps": n,
            "ms_per_step": ms / n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "parallax_step_host", "head_groups": chunks}


def run_case(args):
    """One extra workload alone on cuda:0 (inputs resident in HBM), printed as
    a JSON line of its own figures; not the benchmark line."""
    import torch
    import parallax_local_linear_fwd_b300 as plx

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    if args.case == "fwd_c3":
        res = forward_workload(torch, plx, "c3", dev, stream, iters=args.steps, warmup=args.warmup)
    elif args.case == "probe_c3":
        res = probe_workload(torch, plx, "c3", dev, stream, iters=args.steps, warmup=args.warmup)
    else:
        w = plx_synth.WORKLOADS["c4"]
        inp = plx_synth.generate_workload("c4")
        k, v, P = (torch.from_numpy(inp[x].view(np.int16)).view(torch.bfloat16).to(dev) if inp[x].dtype == np.uint16
                   else torch.from_numpy(inp[x]).to(dev) for x in ("k", "v", "P"))
        res = decode_workload(torch, plx, k, v, P, stream, iters=args.steps, warmup=args.warmup,
                              probe=args.case == "decode_probe")
    code, detail = plx.parallax_last_device_error(stream)
    if code != plx.PLX_OK:
        raise RuntimeError(f"device watchdog: {plx.parallax_strerror(code)} detail={detail:#x}")
    print(json.dumps({"case": args.case, **res}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4", choices=["c4"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fwd-c3", action="store_true",
                    help="skip the extra measurements: the B4 H16 T4096 d128 forward and the decode step")
    ap.add_argument("--shard", default="heads", choices=["heads", "batch"],
                    help="heads: every rank runs its own independent set of heads (no collective); batch: "
                         "the ranks split one problem's batch and all-reduce dP_h each step")
    ap.add_argument("--case", default="step", choices=["step", "fwd_c3", "probe_c3", "decode", "decode_probe"],
                    help="step: the benchmark (default). The others run one of the extra workloads alone "
                         "and print its figures (used for profiling a single kernel family)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps, reported as run
    world, rank, _ = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.case != "step":
        run_case(args)
    else:
        run_ours(args, world, rank)


if __name__ == "__main__":
    main()
