"""Benchmark of the batch-invariant mHC pre "H Aggregate" on GB300.

One step = one pass of the whole hot path over one batch: the forward
(out = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3))) and the fused backward
(grad_residual, grad_pre) on T=4096 tokens of H=7168, inputs resident in HBM.
Bytes per step are the algorithmic ones: T*(10H+16) for the forward and
T*(18H+32) for the backward ("Add batch-invariant h_aggregate kernel",
Performance: GB/s = T*(10H+16)/time for the forward).

Prints one JSON line on rank 0.  Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU runs (torchrun, one rank per GPU) shard by giving every rank its own
batch (weak scaling, no data exchange); only the timing uses a collective.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "h_aggregate fwd/bwd HBM GB/s (% of GB300 peak) and µs/call per (T,H)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 256 << 20

FWD_SWEEP = [("fwd_decode", 2, "decode", [(1, 4096), (8, 4096), (128, 4096),
                                          (1, 7168), (8, 7168), (128, 7168)]),
             ("fwd_prefill", 3, "normal", [(1024, 7168), (4096, 7168), (16384, 7168),
                                           (65536, 7168)])]
BWD_SWEEP = [("bwd_t4096_h7168", 4, "normal", [(4096, 7168)])]


#: the kernel each path of the forward / backward runs
KERNEL_OF_PATH = {
    "fwd": {"vec32": "agg_fwd_vec_kernel", "vec16": "agg_fwd_vec_kernel", "pair": "agg_fwd_pair_kernel",
            "element": "agg_fwd_element_kernel", "shift16": "agg_fwd_shift_kernel"},
    "bwd": {"vec32": "agg_bwd_vec_kernel", "vec16": "agg_bwd_vec_kernel", "pair": "agg_bwd_staged_kernel",
            "element": "agg_bwd_staged_kernel", "shift16": "agg_bwd_shift_kernel"},
}


def fwd_bytes(T, H):
    return T * (10 * H + 16)


def bwd_bytes(T, H):
    return T * (18 * H + 32)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 8000; 3 with --profile-family)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--H", type=int, default=7168)
    ap.add_argument("--phase", choices=("both", "fwd", "bwd"), default="both",
                    help="profiling aid: time only one kernel per step")
    ap.add_argument("--flush", action="store_true",
                    help="flush L2 (write a 256 MiB buffer) before every step; by default the "
                         "step's inputs (larger than L2) are relied on instead")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target length of the CPU oracle baseline sample")
    prof = ap.add_argument_group(
        "profiling workload",
        "--profile-family F runs --steps steps (one warm-up step first) of one call family on "
        "seeded inputs with nothing else in the process, a fixed workload for ncu -k, and prints "
        "one plain line with the mean step time instead of the JSON line.  Families (a step is "
        "the forward then the backward): plain (mhc_aggregate_fwd/bwd), sigmoid "
        "(mhc_aggregate_sigmoid_fwd/bwd, then mhc_sigmoid_param_grad), post (mhc_post_fwd/bwd), "
        "post_sigmoid (mhc_post_sigmoid_fwd/bwd, then mhc_sigmoid_param_grad).  Buffers are "
        "PyTorch allocations, so the path follows from H (H % 16 == 0: 32-byte vectors, "
        "H % 8 == 0: 16-byte, even H: 4-byte pairs, odd H: realigned 16-byte); --offset 2 moves "
        "every 2-byte buffer off its allocation's alignment (the realigned path for H >= 64)")
    prof.add_argument("--profile-family", choices=("plain", "sigmoid", "post", "post_sigmoid"),
                      default=None)
    prof.add_argument("--n", type=int, default=4, help="stream count of the profiling workload")
    prof.add_argument("--dtype", choices=("bf16", "f16"), default="bf16",
                      help="storage type of the profiling workload")
    prof.add_argument("--offset", type=int, default=0,
                      help="byte offset (even) of every 2-byte buffer of the profiling workload")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (the step time every rank waits for)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def stored_traffic(kernel: str, digest: str):
    """DRAM bytes per launch from an ncu capture (profiles/dram_traffic.txt),
    only if it was taken on these exact kernels (same kernel digest)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel:
                lib_digest, T, H = parts[1], parts[2], parts[3]
                bytes_per_launch = float(parts[4])
                if lib_digest == digest[:16]:
                    return bytes_per_launch, int(T), int(H)
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        if not rows:
            return None
        window = [r for r in rows if self.t0 - 0.1 <= r[0] <= self.t1 + 0.3]
        in_window = len(window)
        if not window:
            window = [min(rows, key=lambda r: abs(r[0] - (self.t0 + self.t1) / 2))]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for _, p in window if num(p[2]) is not None]
        smax = [num(p[3]) for _, p in window if num(p[3]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, p in window for i in range(4)
                          if p[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": in_window,
                "power_w_max": max((num(p[4]) or 0.0) for _, p in window)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    from invariant_mhc_aggregate_gb300 import _build, binding
    from invariant_mhc_aggregate_gb300.inputs import backward_inputs, forward_inputs
    from invariant_mhc_aggregate_gb300.sharding import token_range

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=dev)
        dist = dist_mod

    _build.build()
    binding.load()
    digest = _build.kernel_digest()
    T, H = args.T, args.H
    # Weak scaling: rank r owns tokens token_range(world*T, r, world) of a global
    # batch of world*T tokens and draws them with its own seed; no data moves
    # between ranks.
    t_start, t_stop = token_range(world * T, rank, world)
    assert t_stop - t_start == T
    g, res, pre = backward_inputs(T, H, "normal", seed=4 + rank, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    grad_res = torch.empty((T, 4, H), dtype=torch.bfloat16, device=dev)
    grad_pre = torch.empty((T, 4), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    do_fwd = args.phase in ("both", "fwd")
    do_bwd = args.phase in ("both", "bwd")

    def step():
        if do_fwd:
            binding.mhc_h_aggregate_fwd(res, pre, out, stream)
        if do_bwd:
            binding.mhc_h_aggregate_bwd(g, res, pre, grad_res, grad_pre, stream)

    for _ in range(max(args.warmup, 0)):
        if args.flush:
            flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.5)
    # The timed region: K steps back to back, CUDA events only at its two ends
    # (an event between two kernels would stop the second from becoming
    # resident while the first drains).
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    wall0 = time.perf_counter()
    e_start.record(stream)
    for _ in range(K):
        if args.flush:
            flush.zero_()
        step()
    e_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    sampler.mark_end()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop() if rank == 0 else None
    region_ms = e_start.elapsed_time(e_end)
    if args.flush:
        region_ms = None  # the flushes are inside; use the per-kernel pass below

    # Per-kernel pass (for the roofline): the same steps with an event pair
    # around every kernel, on the launching stream.
    K2 = min(K, 500)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    for i in range(K2):
        if args.flush:
            flush.zero_()
        e0, e1, e2 = ev[i]
        e0.record(stream)
        if do_fwd:
            binding.mhc_h_aggregate_fwd(res, pre, out, stream)
        e1.record(stream)
        if do_bwd:
            binding.mhc_h_aggregate_bwd(g, res, pre, grad_res, grad_pre, stream)
        e2.record(stream)
    torch.cuda.synchronize()
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K2)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K2)]
    step_ms_local = region_ms / K if region_ms is not None else (sum(fwd_ms) + sum(bwd_ms)) / K2
    step_ms = max_over_ranks(step_ms_local, dist, dev)

    bytes_step = (fwd_bytes(T, H) if do_fwd else 0) + (bwd_bytes(T, H) if do_bwd else 0)
    value = bytes_step * world / (step_ms * 1e-3) / 1e9

    peak, peak_kind = measured_peaks()
    fwd_us = 1e3 * statistics.fmean(fwd_ms) if do_fwd else None
    bwd_us = 1e3 * statistics.fmean(bwd_ms) if do_bwd else None
    per_kernel = {}
    fwd_path = binding.PATH_NAMES[binding.mhc_h_aggregate_fwd_path(res, pre, out)]
    bwd_path = binding.PATH_NAMES[binding.mhc_h_aggregate_bwd_path(g, res, pre, grad_res, grad_pre)]
    if do_fwd:
        a = fwd_bytes(T, H) / (fwd_us * 1e-6) / 1e9
        per_kernel[KERNEL_OF_PATH["fwd"][fwd_path]] = {"path": fwd_path,"us_mean": round(fwd_us, 3),
                                         "us_p50": round(1e3 * statistics.median(fwd_ms), 3),
                                         "GBps": round(a, 1), "frac": round(a / peak, 4),
                                         "bytes": fwd_bytes(T, H)}
    if do_bwd:
        a = bwd_bytes(T, H) / (bwd_us * 1e-6) / 1e9
        per_kernel[KERNEL_OF_PATH["bwd"][bwd_path]] = {"path": bwd_path,"us_mean": round(bwd_us, 3),
                                         "us_p50": round(1e3 * statistics.median(bwd_ms), 3),
                                         "GBps": round(a, 1), "frac": round(a / peak, 4),
                                         "bytes": bwd_bytes(T, H)}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["us_mean"])
    dk = per_kernel[dom]
    traffic = stored_traffic(dom, digest)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": dk["GBps"], "peak": peak,
                "peak_kind": f"of {peak_kind}", "unit": "GB/s", "frac": dk["frac"],
                "traffic": None, "algorithmic_bytes": dk["bytes"]}
    if traffic is not None:
        tb, tT, tH = traffic
        roofline["traffic"] = round(tb * (T / tT) * (H / tH))
        roofline["traffic_note"] = f"ncu dram bytes at T={tT},H={tH}, scaled by tokens" \
            if (tT, tH) != (T, H) else "ncu dram bytes, same workload"

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"h_aggregate fwd+bwd, T={T}, H={H}" if args.phase == "both"
                   else f"h_aggregate {args.phase} only, T={T}, H={H}",
                   "T": T, "H": H, "tokens_per_rank": T, "global_tokens": world * T,
                   "values": "residual, g ~ N(0,1) rounded to bf16; pre ~ U(0,1); seed 4+rank",
                   "storage": "bf16 residual/out/g/grad_residual, f32 pre/grad_pre",
                   "l2": ("flushed before every step (256 MiB write, outside the timed events)"
                          if args.flush else
                          "not flushed: the step reads 294 MB of inputs (> 126 MB L2) in token "
                          "order, so no kernel finds its inputs in L2"),
                   "timing": ("CUDA events on the launching stream at the two ends of the K-step "
                              "region; per-kernel times (per_kernel, roofline) from a second pass "
                              "of min(K, 500) steps with events around every kernel"),
                   "bytes_per_step": bytes_step},
        "gpu_launches": K * (int(do_fwd) + int(do_bwd)),
        "roofline": roofline,
        "per_kernel": per_kernel,
        "wall_s_timed_region": round(wall, 3),
        "library": {"so": os.path.relpath(_build.LIB_PATH, ROOT),
                    "digest": _build.source_digest()[:16], "kernel_digest": digest[:16]},
    }
    if clocks is not None:
        line["clocks"] = clocks

    if not args.no_e2e:
        line["e2e"] = e2e_measure(args, torch, binding, g, res, pre, dev, stream, world, dist)

    if not args.no_sweep and rank == 0:
        line["sweep"] = sweep(torch, binding, forward_inputs, backward_inputs, dev, flush, peak)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(g, res, pre, T, H, args.cpu_seconds)

    if "sweep" in line:
        # kept last, so that it stays in the tail of a truncated log
        line["kernels_at_h7168"] = headline_kernels(line["sweep"])

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def headline_kernels(results):
    """The forward alone at T = 4096, 16384 and 65536 and the backward alone
    at T = 4096 (H = 7168), from the sweep: steady (back to back, no L2
    reuse), cold_clean (graph replay after an L2 flush that leaves no dirty
    lines) and cold_write_flush (the pages' write flush, whose write-back the
    call pays); microseconds and the fraction of the measured copy peak (m)
    and of 8 TB/s (n)."""
    out = {}
    for e in results:
        key = (e.get("dir"), e.get("T"), e.get("H"))
        if e.get("workload") not in ("fwd_prefill", "bwd_t4096_h7168") or key not in (
                ("fwd", 4096, 7168), ("fwd", 16384, 7168), ("fwd", 65536, 7168), ("bwd", 4096, 7168)):
            continue
        d = {}
        for col, name in (("steady", "steady"), ("cold_clean", "cold_clean"),
                          ("cold", "cold_write_flush")):
            if col not in e:
                continue
            c = e[col]
            us = c["us"] if "us" in c else c["us_p20_p50_p80"][1]
            d[name] = {"us": us, "m": c["frac_of_measured"], "n": c["frac_of_8TBs"]}
        out[f"{key[0]}_t{key[1]}"] = d
    return out


def e2e_measure(args, torch, binding, g, res, pre, dev, stream, world, dist):
    """The step through the public API with host buffers: pinned host inputs,
    forward, backward and pinned host outputs, all inside the timed region.
    The library's HostPipeline splits the batch into token chunks and overlaps
    host -> device copies, the kernels and device -> host copies on three
    streams (tokens are independent, so the bytes are those of one call)."""
    from invariant_mhc_aggregate_gb300.pipeline import HostPipeline
    T, H = args.T, args.H
    hg = g.cpu().pin_memory()
    hr = res.cpu().pin_memory()
    hp = pre.cpu().pin_memory()
    ho = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    hgr = torch.empty((T, 4, H), dtype=torch.bfloat16).pin_memory()
    hgp = torch.empty((T, 4), dtype=torch.float32).pin_memory()
    pipe = HostPipeline(4, H, torch.bfloat16, chunk_tokens=min(1024, T), slots=5, device=dev)
    # the first steps on fresh pinned buffers run up to 30% slower (measured:
    # 2.5 against 1.94 ms a step at T=4096 with 512-token chunks), so warm up
    # for several steps
    for _ in range(10):
        pipe.step(hr, hp, hg, ho, hgr, hgp)
    pipe.synchronize()
    n = max(5, min(args.steps, 50))
    # five rounds of n steps, the median round reported: the host link's
    # rate varies from round to round (1.82 to 3.10 ms a step seen on one box)
    rounds = []
    for _ in range(5):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(pipe.h2d)
        for _ in range(n):
            pipe.step(hr, hp, hg, ho, hgr, hgp)
        e1.record(pipe.d2h)
        torch.cuda.synchronize()
        rounds.append(e0.elapsed_time(e1) / n)
    ms = max_over_ranks(sorted(rounds)[len(rounds) // 2], dist, dev)
    # the host results are the device results of the same inputs
    d_out = binding.h_aggregate(res, pre)
    d_gr, d_gp = binding.h_aggregate_backward(g, res, pre)
    assert torch.equal(hgp, d_gp.cpu()) and torch.equal(ho.view(torch.int16), d_out.cpu().view(torch.int16))
    assert torch.equal(hgr.view(torch.int16), d_gr.cpu().view(torch.int16))
    h2d = hr.numel() * 2 + hp.numel() * 4 + hg.numel() * 2
    d2h = ho.numel() * 2 + hgr.numel() * 2 + hgp.numel() * 4
    value = (fwd_bytes(T, H) + bwd_bytes(T, H)) * world / (ms * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "rounds_ms": [round(r, 4) for r in rounds],
            "note": ("pinned host buffers; HostPipeline: 1024-token chunks in 5 slots, host->device copies, "
                     "kernels and device->host copies overlapped on three streams")}


def sweep(torch, binding, forward_inputs, backward_inputs, dev, flush, peak):
    """us/call per (T,H).

    "cold": CUDA-graph replay of one call with L2 flushed by a 256 MiB write
    before each sample (the pages' cold-L2 method); 7 rounds x (10 warm-up +
    100 samples), p20/p50/p80 of the round medians.  The write flush leaves
    up to a whole L2 of dirty lines that the timed call has to write back, so
    this column charges the flush's own write-back to the call.
    "cold_clean": the same, with a read of 4x L2 after the write flush and
    before the start event: the flush's dirty lines are written back during
    that read, and the timed call starts with an L2 holding only clean lines
    of an unrelated buffer (none of its inputs, nothing to write back).
    "steady": about 400 calls back to back (a CUDA graph of at least 16
    calls, replayed), rotating over enough buffer sets that no call finds its
    inputs in L2 (at least 3x L2 in total), events only at the two ends;
    shapes whose sets would not reach that in 8 sets get a "warm" entry
    instead (16 sets that stay in L2, as a decode step's freshly written
    inputs would).
    """
    results = []
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    rflush = torch.ones(4 * l2 // 8, dtype=torch.int64, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def time_graph(graph, clean=False):
        meds = []
        for _ in range(7):
            samples = []
            for i in range(110):
                flush.zero_()
                if clean:
                    torch.sum(rflush, dim=0, out=sink)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                graph.replay()
                e1.record()
                e1.synchronize()
                samples.append((e0, e1))
            ts = [a.elapsed_time(b) * 1e3 for a, b in samples[10:]]
            meds.append(statistics.median(ts))
        q = np.quantile(np.array(meds), [0.2, 0.5, 0.8])
        return [round(float(x), 3) for x in q]

    def time_steady(call, sets, n=400):
        """Per-call time of back-to-back calls rotating over `sets`, from a CUDA
        graph of at least 16 calls (so the host's launch cost is out of the
        measurement and consecutive kernels keep their programmatic overlap),
        replayed until about n calls ran; events only at the two ends."""
        per_graph = max(16, len(sets))
        for i in range(len(sets)):
            call(*sets[i])
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(per_graph):
                call(*sets[i % len(sets)])
        reps = max(2, n // per_graph)
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        del graph
        return round(e0.elapsed_time(e1) * 1e3 / (reps * per_graph), 3)

    def entry_for(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"GBps": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4)}

    def n_sets(set_bytes):
        n = max(2, -(-3 * l2 // set_bytes))
        return n if n <= 8 else None

    # The floor of the cold method: a graph holding one trivial kernel.
    z = torch.zeros(1, device=dev)
    floor_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(floor_graph, stream=stream):
        z.add_(1.0)
    results.append({"workload": "launch_floor", "dir": "none",
                    "note": "one trivial kernel timed by the cold method (graph replay after a "
                            "256 MiB write flush, CUDA events)",
                    "cold": {"us_p20_p50_p80": time_graph(floor_graph)},
                    "cold_clean": {"us_p20_p50_p80": time_graph(floor_graph, clean=True)}})
    del floor_graph

    for name, seed, recipe, shapes in FWD_SWEEP:
        for T, H in shapes:
            r, p = forward_inputs(T, H, recipe, seed, device=dev)
            o = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            binding.mhc_h_aggregate_fwd(r, p, o)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                binding.mhc_h_aggregate_fwd(r, p, o)
            nbytes = fwd_bytes(T, H)
            us = time_graph(graph)
            us_c = time_graph(graph, clean=True)
            entry = {"workload": name, "dir": "fwd", "T": T, "H": H,
                     "cold": {"us_p20_p50_p80": us, **entry_for(us[1], nbytes)},
                     "cold_clean": {"us_p20_p50_p80": us_c, **entry_for(us_c[1], nbytes)}}
            del graph
            ns = n_sets(nbytes)
            if ns is not None:
                sets = [(r, p, o)] + [(torch.empty_like(r).copy_(r), p.clone(), torch.empty_like(o))
                                      for _ in range(ns - 1)]
                us_s = time_steady(lambda a, b, c: binding.mhc_h_aggregate_fwd(a, b, c), sets)
                entry["steady"] = {"us": us_s, "sets": ns, **entry_for(us_s, nbytes)}
                del sets
            elif T <= 128:
                # decode-sized: back-to-back calls over 16 buffer sets that stay in L2
                # (as a decode step's inputs, just written by the previous layer, would)
                sets = [(r, p, o)] + [(torch.empty_like(r).copy_(r), p.clone(), torch.empty_like(o))
                                      for _ in range(15)]
                us_w = time_steady(lambda a, b, c: binding.mhc_h_aggregate_fwd(a, b, c), sets)
                entry["warm"] = {"us": us_w, "sets": 16, "note": "back-to-back, inputs L2-resident",
                                 **entry_for(us_w, nbytes)}
                del sets
            results.append(entry)
            del r, p, o
            torch.cuda.empty_cache()
    for name, seed, recipe, shapes in BWD_SWEEP:
        for T, H in shapes:
            g, r, p = backward_inputs(T, H, recipe, seed, device=dev)
            gr = torch.empty((T, 4, H), dtype=torch.bfloat16, device=dev)
            gp = torch.empty((T, 4), dtype=torch.float32, device=dev)
            binding.mhc_h_aggregate_bwd(g, r, p, gr, gp)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                binding.mhc_h_aggregate_bwd(g, r, p, gr, gp)
            nbytes = bwd_bytes(T, H)
            us = time_graph(graph)
            us_c = time_graph(graph, clean=True)
            entry = {"workload": name, "dir": "bwd", "T": T, "H": H,
                     "cold": {"us_p20_p50_p80": us, **entry_for(us[1], nbytes)},
                     "cold_clean": {"us_p20_p50_p80": us_c, **entry_for(us_c[1], nbytes)}}
            del graph
            ns = n_sets(nbytes)
            if ns is not None:
                sets = [(g, r, p, gr, gp)] + [(g.clone(), r.clone(), p.clone(), torch.empty_like(gr),
                                               torch.empty_like(gp)) for _ in range(ns - 1)]
                us_s = time_steady(lambda a, b, c, d, e: binding.mhc_h_aggregate_bwd(a, b, c, d, e), sets)
                entry["steady"] = {"us": us_s, "sets": ns, **entry_for(us_s, nbytes)}
                del sets
            results.append(entry)
            del g, r, p, gr, gp
            torch.cuda.empty_cache()
    # the narrow paths (H even but not a multiple of 8: 4-byte; H odd: 2-byte), steady state
    for H in (7166, 7167):
        T = 4096
        g, r, p = backward_inputs(T, H, "normal", 4, device=dev)
        sets = [(g, r, p), (g.clone(), r.clone(), p.clone())]
        fsets = [(rr, pp, torch.empty((T, H), dtype=torch.bfloat16, device=dev)) for _, rr, pp in sets]
        bsets = [(gg, rr, pp, torch.empty_like(rr), torch.empty_like(pp)) for gg, rr, pp in sets]
        fpath = binding.PATH_NAMES[binding.mhc_h_aggregate_fwd_path(*fsets[0])]
        bpath = binding.PATH_NAMES[binding.mhc_h_aggregate_bwd_path(*bsets[0])]
        us_f = time_steady(lambda a, b, c: binding.mhc_h_aggregate_fwd(a, b, c), fsets)
        us_b = time_steady(lambda a, b, c, d, e: binding.mhc_h_aggregate_bwd(a, b, c, d, e), bsets)
        results.append({"workload": f"narrow_h{H}", "dir": "fwd", "T": T, "H": H, "path": fpath,
                        "steady": {"us": us_f, "sets": 2, **entry_for(us_f, fwd_bytes(T, H))}})
        results.append({"workload": f"narrow_h{H}", "dir": "bwd", "T": T, "H": H, "path": bpath,
                        "steady": {"us": us_b, "sets": 2, **entry_for(us_b, bwd_bytes(T, H))}})
        del g, r, p, sets, fsets, bsets
        torch.cuda.empty_cache()

    # the general form (stream count n, FP16 storage), steady state only
    for n, dtype in ((8, torch.bfloat16), (2, torch.bfloat16), (4, torch.float16)):
        T, H = 4096, 7168
        name = f"general_n{n}_{'bf16' if dtype == torch.bfloat16 else 'f16'}"
        g, r, p = backward_inputs(T, H, "normal", 4, device=dev, n=n, dtype=dtype)
        fb = T * (2 * (n + 1) * H + 4 * n)
        bb = T * (2 * (2 * n + 1) * H + 8 * n)
        sets = [(g, r, p)] + [(g.clone(), r.clone(), p.clone()) for _ in range(max(1, n_sets(fb) or 2) - 1)]
        fsets = [(rr, pp, torch.empty((T, H), dtype=dtype, device=dev)) for _, rr, pp in sets]
        us_f = time_steady(lambda a, b, c: binding.mhc_aggregate_fwd(a, b, c), fsets)
        bsets = [(gg, rr, pp, torch.empty_like(rr), torch.empty((T, n), dtype=torch.float32, device=dev))
                 for gg, rr, pp in sets]
        us_b = time_steady(lambda a, b, c, d, e: binding.mhc_aggregate_bwd(a, b, c, d, e), bsets)
        results.append({"workload": name, "dir": "fwd", "T": T, "H": H, "n": n,
                        "steady": {"us": us_f, "sets": len(sets), **entry_for(us_f, fb)}})
        results.append({"workload": name, "dir": "bwd", "T": T, "H": H, "n": n,
                        "steady": {"us": us_b, "sets": len(sets), **entry_for(us_b, bb)}})
        del g, r, p, sets, fsets, bsets
        torch.cuda.empty_cache()

    # pre computed in the kernels from the mix (sigmoid of alpha * mix + b), n = 4 BF16,
    # steady state; and the reduction of grad_b / grad_alpha over the tokens
    from invariant_mhc_aggregate_gb300.inputs import coeff_inputs
    T, H = 4096, 7168
    g, r, _ = backward_inputs(T, H, "normal", 4, device=dev)
    mix, alpha, b = coeff_inputs(T, 4, "normal", 5, device=dev)
    fb = T * (10 * H + 16)
    bb = T * (18 * H + 48)
    ns = n_sets(fb) or 2
    sets = [(g, r, mix)] + [(g.clone(), r.clone(), mix.clone()) for _ in range(ns - 1)]
    fsets = [(rr, mm, alpha, b, torch.empty((T, H), dtype=torch.bfloat16, device=dev))
             for _, rr, mm in sets]
    us_f = time_steady(lambda *a: binding.mhc_aggregate_sigmoid_fwd(*a), fsets)
    bsets = [(gg, rr, mm, alpha, b, torch.empty_like(rr), torch.empty_like(mm), torch.empty_like(mm))
             for gg, rr, mm in sets]
    us_b = time_steady(lambda *a: binding.mhc_aggregate_sigmoid_bwd(*a), bsets)
    psets = [(bs[6], bs[2], torch.empty(4, device=dev), torch.empty(1, device=dev)) for bs in bsets]
    us_p = time_steady(lambda *a: binding.mhc_sigmoid_param_grad(*a), psets)
    results.append({"workload": "sigmoid_coeffs_n4_bf16", "dir": "fwd", "T": T, "H": H,
                    "note": "pre = sigmoid(alpha*mix + b) computed in the kernel; bytes T*(10H+16)",
                    "steady": {"us": us_f, "sets": ns, **entry_for(us_f, fb)}})
    results.append({"workload": "sigmoid_coeffs_n4_bf16", "dir": "bwd", "T": T, "H": H,
                    "note": "grad_residual, grad_z, grad_mix; bytes T*(18H+48)",
                    "steady": {"us": us_b, "sets": ns, **entry_for(us_b, bb)}})
    results.append({"workload": "sigmoid_param_grad_n4", "dir": "bwd", "T": T,
                    "note": "grad_b and grad_alpha summed over the tokens (one cluster of 8 CTAs); "
                            "bytes T*32, latency-bound",
                    "steady": {"us": us_p, "sets": ns}})
    del g, r, mix, sets, fsets, bsets, psets
    torch.cuda.empty_cache()

    # the mHC post (the layer output expanded back onto the n streams), steady state
    from invariant_mhc_aggregate_gb300.inputs import post_inputs
    for n in (1, 2, 4, 8):
        T, H = 4096, 7168
        x, y, post, res, g = post_inputs(T, H, n, "normal", 6, device=dev, with_grad=True)
        fb = T * (2 * (2 * n + 1) * H + 4 * n + 4 * n * n)
        bb = T * (2 * (3 * n + 2) * H + 8 * n + 8 * n * n)
        ns = n_sets(fb) or 2
        sets = [(g, x, y, post, res)] + [tuple(t.clone() for t in (g, x, y, post, res))
                                         for _ in range(ns - 1)]
        fsets = [(xx, yy, pp, rr, torch.empty_like(xx)) for _, xx, yy, pp, rr in sets]
        fpath = binding.PATH_NAMES[binding.post_fwd_path_raw(*(t.data_ptr() for t in fsets[0]), T, n, H)]
        us_f = time_steady(lambda *a: binding.mhc_post_fwd(*a), fsets)
        del fsets
        bsets = [(gg, xx, yy, pp, rr, torch.empty_like(xx), torch.empty_like(yy), torch.empty_like(pp),
                  torch.empty_like(rr)) for gg, xx, yy, pp, rr in sets]
        bpath = binding.PATH_NAMES[binding.post_bwd_path_raw(*(t.data_ptr() for t in bsets[0]), T, n, H)]
        us_b = time_steady(lambda *a: binding.mhc_post_bwd(*a), bsets)
        results.append({"workload": f"post_n{n}_bf16", "dir": "fwd", "T": T, "H": H, "n": n, "path": fpath,
                        "note": "out = tree(res*x) + post*y; bytes T*(2(2n+1)H + 4n + 4n^2)",
                        "steady": {"us": us_f, "sets": ns, **entry_for(us_f, fb)}})
        results.append({"workload": f"post_n{n}_bf16", "dir": "bwd", "T": T, "H": H, "n": n, "path": bpath,
                        "note": "grad_x, grad_y, grad_post, grad_res; bytes T*(2(3n+2)H + 8n + 8n^2)",
                        "steady": {"us": us_b, "sets": ns, **entry_for(us_b, bb)}})
        del x, y, post, res, g, sets, bsets
        torch.cuda.empty_cache()

    # the mHC post with post = sigmoid(alpha * mix + b) computed in the kernels, n = 4
    T, H, n = 4096, 7168, 4
    x, y, _, res, g = post_inputs(T, H, n, "normal", 6, device=dev, with_grad=True)
    mix, alpha, b = coeff_inputs(T, n, "normal", 7, device=dev)
    fb = T * (2 * (2 * n + 1) * H + 4 * n + 4 * n * n)
    bb = T * (2 * (3 * n + 2) * H + 12 * n + 8 * n * n)
    ns = n_sets(fb) or 2
    sets = [(g, x, y, mix, res)] + [tuple(t.clone() for t in (g, x, y, mix, res)) for _ in range(ns - 1)]
    fsets = [(xx, yy, mm, alpha, b, rr, torch.empty_like(xx)) for _, xx, yy, mm, rr in sets]
    us_f = time_steady(lambda *a: binding.mhc_post_sigmoid_fwd(*a), fsets)
    del fsets
    bsets = [(gg, xx, yy, mm, alpha, b, rr, torch.empty_like(xx), torch.empty_like(yy), torch.empty_like(mm),
              torch.empty_like(mm), torch.empty_like(rr)) for gg, xx, yy, mm, rr in sets]
    us_b = time_steady(lambda *a: binding.mhc_post_sigmoid_bwd(*a), bsets)
    results.append({"workload": "post_sigmoid_n4_bf16", "dir": "fwd", "T": T, "H": H, "n": n,
                    "note": "post = sigmoid(alpha*mix + b) computed in the kernel; bytes T*(18H + 80)",
                    "steady": {"us": us_f, "sets": ns, **entry_for(us_f, fb)}})
    results.append({"workload": "post_sigmoid_n4_bf16", "dir": "bwd", "T": T, "H": H, "n": n,
                    "note": "grad_x, grad_y, grad_res, grad_z, grad_mix; bytes T*(28H + 176)",
                    "steady": {"us": us_b, "sets": ns, **entry_for(us_b, bb)}})
    del x, y, res, g, mix, sets, bsets
    torch.cuda.empty_cache()
    torch.cuda.synchronize()
    return results


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def _oracle_pass(o, g_u16, r_u16, pre_f32, threads: int):
    """Forward and backward of the oracle over all tokens given, tokens split
    into contiguous blocks over `threads` host threads (ctypes releases the GIL;
    tokens are independent, so the results do not depend on the split)."""
    T, _, H = r_u16.shape
    out = np.empty((T, H), dtype=np.uint16)
    gr = np.empty((T, 4, H), dtype=np.uint16)
    gp = np.empty((T, 4), dtype=np.float32)
    bounds = np.linspace(0, T, threads + 1).astype(int)

    def work(a, b):
        if b <= a:
            return
        o.lib.oracle_h_aggregate_fwd(r_u16[a:b].ctypes.data, pre_f32[a:b].ctypes.data,
                                     out[a:b].ctypes.data, b - a, H)
        o.lib.oracle_h_aggregate_bwd(g_u16[a:b].ctypes.data, r_u16[a:b].ctypes.data,
                                     pre_f32[a:b].ctypes.data, gr[a:b].ctypes.data,
                                     gp[a:b].ctypes.data, b - a, H)

    ths = [threading.Thread(target=work, args=(int(bounds[i]), int(bounds[i + 1])))
           for i in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    return out, gr, gp


def _host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(g, res, pre, T, H, seconds):
    """The CPU oracle, as it stands, on the host cores over a bounded sample of
    the same workload (whole tokens), sized to about `seconds` of work."""
    import torch
    import oracle

    def host(n_tok):
        return (g[:n_tok].contiguous().cpu().view(torch.int16).numpy().view(np.uint16),
                res[:n_tok].contiguous().cpu().view(torch.int16).numpy().view(np.uint16),
                pre[:n_tok].contiguous().cpu().numpy())

    o = oracle.default()
    threads = _host_threads()
    probe = min(T, 64)
    t0 = time.perf_counter()
    _oracle_pass(o, *host(probe), threads)
    per_token = (time.perf_counter() - t0) / probe
    n_tok = int(min(T, max(probe, seconds / max(per_token, 1e-9))))
    reps = max(1, int(seconds / max(per_token * n_tok, 1e-9)))
    sample = host(n_tok)
    t0 = time.perf_counter()
    for _ in range(reps):
        _oracle_pass(o, *sample, threads)
    dt = time.perf_counter() - t0
    bytes_done = reps * (fwd_bytes(n_tok, H) + bwd_bytes(n_tok, H))
    return {"value": round(bytes_done / dt / 1e9, 3), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} x {n_tok} of {T} tokens (H={H}), forward + backward, "
                      f"{dt:.1f} s on {threads} host threads"}


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, on the same metric
    and workload, each step a bounded sample (256 whole tokens) of the batch."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    import oracle
    from invariant_mhc_aggregate_gb300.inputs import backward_inputs
    T, H = args.T, args.H
    n_tok = min(T, 256)
    g, res, pre = backward_inputs(n_tok, H, "normal", seed=4, device="cpu")
    gu = g.view(torch.int16).numpy().view(np.uint16)
    ru = res.view(torch.int16).numpy().view(np.uint16)
    pf = pre.numpy()
    o = oracle.default()
    threads = _host_threads()
    for _ in range(max(args.warmup, 0)):
        _oracle_pass(o, gu, ru, pf, threads)
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        _oracle_pass(o, gu, ru, pf, threads)
    dt = time.perf_counter() - t0
    bytes_step = fwd_bytes(n_tok, H) + bwd_bytes(n_tok, H)
    value = bytes_step * K / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / K, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"h_aggregate fwd+bwd, T={T}, H={H}", "T": T, "H": H,
                   "sample_tokens_per_step": n_tok,
                   "values": "residual, g ~ N(0,1) rounded to bf16; pre ~ U(0,1); seed 4"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n_tok} of {T} tokens per step, forward + backward"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# profiling workload: one call family, nothing else in the process
# ---------------------------------------------------------------------------

def _shifted(torch, t, offset: int):
    """A copy of t placed `offset` bytes past its allocation's alignment."""
    if offset == 0:
        return t
    n = t.numel()
    buf = torch.empty(n + 256, dtype=t.dtype, device=t.device)
    e = offset // t.element_size()
    view = buf[e:e + n].view(t.shape)
    view.copy_(t)
    return view


def run_profile_family(args):
    import torch
    from invariant_mhc_aggregate_gb300 import _build, binding
    from invariant_mhc_aggregate_gb300.inputs import backward_inputs, coeff_inputs, post_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    if args.offset % 2:
        raise SystemExit("--offset must be even (2-byte elements)")
    _build.build()
    binding.load()
    dev = torch.device("cuda", 0)
    dtype = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    T, H, n, fam = args.T, args.H, args.n, args.profile_family
    sh = lambda t: _shifted(torch, t, args.offset)  # noqa: E731
    ptrs = lambda *ts: [t.data_ptr() for t in ts]  # noqa: E731
    if fam in ("post", "post_sigmoid"):
        x, y, post, res, g = post_inputs(T, H, n, "normal", 6, device=dev, dtype=dtype, with_grad=True)
        x, y, g = sh(x), sh(y), sh(g)
        out, gx, gy = sh(torch.empty_like(x)), sh(torch.empty_like(x)), sh(torch.empty_like(y))
        gp, gr = torch.empty_like(post), torch.empty_like(res)
        paths = (binding.post_fwd_path_raw(*ptrs(x, y, post, res, out), T, n, H),
                 binding.post_bwd_path_raw(*ptrs(g, x, y, post, res, gx, gy, gp, gr), T, n, H))
        if fam == "post":
            def step():
                binding.mhc_post_fwd(x, y, post, res, out)
                binding.mhc_post_bwd(g, x, y, post, res, gx, gy, gp, gr)
        else:
            mix, alpha, b = coeff_inputs(T, n, "normal", 7, device=dev)
            gm = torch.empty_like(mix)
            gb = torch.empty((n,), dtype=torch.float32, device=dev)
            ga = torch.empty((1,), dtype=torch.float32, device=dev)

            def step():
                binding.mhc_post_sigmoid_fwd(x, y, mix, alpha, b, res, out)
                binding.mhc_post_sigmoid_bwd(g, x, y, mix, alpha, b, res, gx, gy, gp, gm, gr)
                binding.mhc_sigmoid_param_grad(gp, mix, gb, ga)
    else:
        g, res, pre = backward_inputs(T, H, "normal", 4, device=dev, n=n, dtype=dtype)
        g, res = sh(g), sh(res)
        out = sh(torch.empty((T, H), dtype=dtype, device=dev))
        gres = sh(torch.empty((T, n, H), dtype=dtype, device=dev))
        if fam == "plain":
            coef = pre
            gp = torch.empty((T, n), dtype=torch.float32, device=dev)

            def step():
                binding.mhc_aggregate_fwd(res, pre, out)
                binding.mhc_aggregate_bwd(g, res, pre, gres, gp)
        else:
            mix, alpha, b = coeff_inputs(T, n, "normal", 5, device=dev)
            coef = mix
            gp = torch.empty((T, n), dtype=torch.float32, device=dev)
            gm = torch.empty_like(gp)
            gb = torch.empty((n,), dtype=torch.float32, device=dev)
            ga = torch.empty((1,), dtype=torch.float32, device=dev)

            def step():
                binding.mhc_aggregate_sigmoid_fwd(res, mix, alpha, b, out)
                binding.mhc_aggregate_sigmoid_bwd(g, res, mix, alpha, b, gres, gp, gm)
                binding.mhc_sigmoid_param_grad(gp, mix, gb, ga)
        paths = (binding.agg_fwd_path_raw(*ptrs(res, coef, out), T, n, H),
                 binding.agg_bwd_path_raw(*ptrs(g, res, coef, gres, gp), T, n, H))
    step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / max(args.steps, 1)
    print(f"{fam} T={T} H={H} n={n} {args.dtype} offset={args.offset} paths fwd/bwd="
          f"{binding.PATH_NAMES[paths[0]]}/{binding.PATH_NAMES[paths[1]]}: {us:.1f} us per step",
          flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.steps is None:
        args.steps = 3 if args.profile_family is not None else 8000
    if args.profile_family is not None:
        run_profile_family(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
