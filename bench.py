"""Benchmark of one continuous-batching decode step over a paged KV cache.

A step is the whole hot path over one batch: the newest-token slot mapping,
then for every layer the KV append and the paged decode attention.  The
headline workload is the Llama-3-8B-shaped batch-32 step: 32 layers, 32
sequences of 4096 tokens (the appended token included), 32 query / 8 KV
heads, head_dim 128, bf16 K/V, 16-token blocks, a 16384-block pool per layer.

Timed region: exactly K graph replays of the captured step, bracketed by a
barrier and a device synchronize, CUDA events on the replay stream, max over
ranks.  The region is repeated until the regions add up to a floor of device
time (--min-timed-ms); the value is the bytes of all timed steps over the
summed time.  One step reads 17.2 GB of K/V, far above the 129 MB L2, so no
flush is needed.

After the headline, the same line carries a `configs` object: every other
workload (the tiny check case, the one-layer batch-8 step, the mixed-length
prefix-sharing step, the batch-256 serving step, the E4M3 variants, the
chunked-prefill step and the swap copies), each timed the same way.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host cores instead (bounded samples of the same workload).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import SPECS, fill_pool_layer, make_placement, pool_layer_values, step_layer_values  # noqa: E402

METRIC = "paged decode-attention KV GB/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SOURCES = ("decode_kernel.cuh", "decode_mma.cu", "decode_ffma.cu", "decode_fp8.cu", "mma_frag.cuh",
                  "device_utils.cuh", "decode_plan.cu")
L2_BYTES = 129 * 10**6  # GB300 L2
PREFILL_SOURCES = ("prefill_tc.cu", "prefill.cu", "tc_utils.cuh", "decode_kernel.cuh", "mma_frag.cuh",
                   "device_utils.cuh")
# Workloads of the `configs` object, in the order they run (the headline's
# own workload is skipped there).  "swap" is the block swap copies.
CONFIG_ORDER = ("tiny", "llama8b_layer_b8", "mixed_prefix_b64", "serving_b256", "llama8b_32l_b32_fp8",
                "serving_b256_fp8", "chunked_prefill_b32", "swap")
BACK_TO_BACK_POOLS = 8  # independent layer pools of the rotated one-layer measurement


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama8b_32l_b32", choices=sorted(SPECS))
    p.add_argument("--configs", default="all",
                   help="workloads measured after the headline: 'all', 'none' or a comma list of "
                        + ", ".join(CONFIG_ORDER))
    p.add_argument("--min-timed-ms", type=float, default=1000.0,
                   help="floor on the headline's summed timed device time (regions of exactly K steps)")
    p.add_argument("--config-min-timed-ms", type=float, default=300.0,
                   help="the same floor for every entry of `configs`")
    p.add_argument("--kernel", default="auto", choices=["auto", "mma", "ffma"])
    p.add_argument("--consumer-warps", type=int, default=0, help="0: library default")
    p.add_argument("--ctas-per-sm", type=int, default=0, help="0: library default")
    p.add_argument("--heads-per-stage", type=int, default=0, help="0: library default")
    p.add_argument("--separate-reduce", action="store_true")
    p.add_argument("--no-pdl", action="store_true")
    p.add_argument("--no-early-reads", action="store_true",
                   help="do not let a layer's kernel read tables/cache before the previous layer's kernel ends")
    p.add_argument("--unfused", action="store_true",
                   help="slot mapping + append + attention as separate calls instead of one fused call per layer")
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: run the first N layers (the JSON line then names N)")
    p.add_argument("--swap", action="store_true",
                   help="measure swap-out/in of KV blocks to page-locked host memory instead")
    p.add_argument("--swap-requests", type=int, default=8,
                   help="requests of 2000 tokens (8B shape) swapped per timed copy")
    p.add_argument("--prefill", action="store_true",
                   help="time the multi-token (chunked-prefill) step of --workload chunked_prefill_b32 instead")
    p.add_argument("--block-size", type=int, default=0,
                   help="override the workload's tokens per block (prefill leg; 0: the workload's)")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--cpu-single-seconds", type=float, default=4.0,
                   help="time of the single-thread oracle sample of cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, use_cuda):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if use_cuda else "gloo")


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def timed_regions(run_region, min_ms: float, world: int, device, max_regions: int = 1000) -> list:
    """Time regions until their summed device time reaches `min_ms`.

    run_region() times exactly one region (a fixed number of steps, each
    rank on its own device) and returns its milliseconds; each region's time
    is the max over ranks, so every rank sees the same list and stops after
    the same region."""
    regions = []
    while True:
        barrier(world)
        ms = max_over_ranks(run_region(), world, device)
        barrier(world)
        regions.append(ms)
        if sum(regions) >= min_ms or len(regions) >= max_regions:
            return regions


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_slots_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_name: str, workload: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(sources)
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = dict(kv.split("=", 1) for kv in line.split())
        if f.get("kernel") == kernel_name and f.get("workload") == workload and f.get("sources") == want:
            return int(f["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms meanwhile
    (into a temporary file that is removed afterwards)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"pkv_clocks_{index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
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
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        # Samples under load: the power well above the idle draw of the part.
        p_max = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * p_max] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": p_max, "samples": len(rows), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- our arm
class Step:
    """Device state of a decode workload and one decode step through the library."""

    def __init__(self, spec, kernel, device, fused=True, **opts):
        import paged_kv_cache_slots_gb300 as pkv
        self.pkv = pkv
        self.spec, self.kernel, self.dev, self.fused = spec, kernel, device, fused
        self.opts = dict(kernel=kernel, **opts)
        self.pl = make_placement(spec)
        s, pl = spec, self.pl
        B = len(pl.context_lens)
        self.B = B
        self.pool = pkv.KVPool(s.num_layers, pl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim,
                               s.cache_torch_dtype, device=device)
        self.scales = dict(k_scale=s.kv_scales[0], v_scale=s.kv_scales[1]) if s.fp8 else {}
        self.layers = [self.pool.layer(l) for l in range(s.num_layers)]
        for l, (kc, vc) in enumerate(self.layers):
            fill_pool_layer(s, l, kc, vc)
        self.q = torch.empty((s.num_layers, B, s.num_q_heads, s.head_dim), dtype=s.torch_dtype, device=device)
        self.kn = torch.empty((s.num_layers, B, s.num_kv_heads, s.head_dim), dtype=s.torch_dtype, device=device)
        self.vn = torch.empty_like(self.kn)
        for l in range(s.num_layers):
            q, kn, vn = step_layer_values(s, B, l, device)
            self.q[l].copy_(q)
            self.kn[l].copy_(kn)
            self.vn[l].copy_(vn)
        self.tables = torch.from_numpy(pl.block_tables).to(device)
        self.ctx = torch.from_numpy(pl.context_lens).to(device)
        self.seq_ids = torch.from_numpy(np.where(pl.appends, np.arange(B), -1).astype(np.int32)).to(device)
        self.slots = torch.empty(B, dtype=torch.int32, device=device)
        self.out = torch.empty((s.num_layers, B, s.num_q_heads, s.head_dim), dtype=s.torch_dtype, device=device)
        self.ws = pkv.make_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim, device, **self.opts)
        per_layer = (2 if self.opts.get("separate_reduce") else 1) + (0 if fused else 1)
        self.launches_per_step = (0 if fused else 1) + per_layer * s.num_layers

    def run(self, events=None):
        s, pkv = self.spec, self.pkv
        if not self.fused:
            pkv.slot_mapping(self.tables, self.ctx, s.block_size, self.pl.num_blocks, out=self.slots)
        for l, (kc, vc) in enumerate(self.layers):
            if events is not None:
                events[l][0].record()
            if self.fused:
                pkv.paged_decode_append_attention(self.q[l], self.kn[l], self.vn[l], kc, vc, self.tables,
                                                  self.ctx, s.attn_scale, seq_ids=self.seq_ids,
                                                  out=self.out[l], slot_mapping=self.slots,
                                                  workspace=self.ws, **self.scales, **self.opts)
            else:
                self.pool.append(l, self.kn[l], self.vn[l], self.slots, seq_ids=self.seq_ids, **self.scales)
                pkv.paged_decode_attention(self.q[l], kc, vc, self.tables, self.ctx, s.attn_scale,
                                           out=self.out[l], workspace=self.ws, **self.scales, **self.opts)
            if events is not None:
                events[l][1].record()


def decode_opts(args) -> dict:
    return dict(consumer_warps=args.consumer_warps, ctas_per_sm=args.ctas_per_sm,
                heads_per_stage=args.heads_per_stage, separate_reduce=args.separate_reduce,
                pdl=not args.no_pdl, early_reads=not (args.no_early_reads or args.unfused))


def decode_kernel_name(spec, kernel, fused):
    name = "paged_decode_partial_kernel<MmaPolicy>" if kernel != "ffma" else "paged_decode_partial_kernel<FfmaPolicy>"
    if spec.fp8:
        name = "paged_decode_partial_kernel<MmaFp8Policy>"
    elif spec.dtype == "f32":
        name = "paged_decode_partial_kernel<FfmaPolicy>"
    return name + ("_with_fused_append" if fused else "")


def measure_decode(spec, args, dev, world, min_ms, steps, warmup, kernel="auto", fused=True, opts=None):
    """Capture one decode step of `spec` in a CUDA graph and time it.

    Regions of exactly `steps` replays are timed until they add up to
    `min_ms`.  A step that reads less than 4x the L2 is timed replay by
    replay instead, each after a write of twice the L2 outside the events.
    Returns (result dict, Step)."""
    import paged_kv_cache_slots_gb300 as pkv
    from paged_kv_cache_slots_gb300 import roofline

    opts = dict(opts or {})
    step = Step(spec, kernel, dev, fused=fused, **opts)
    pl = step.pl
    B = step.B
    bytes_layer = roofline.attention_bytes(pl.context_lens, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                           spec.elem_bytes, spec.block_size, spec.elem_bytes,
                                           int(pl.appends.sum()), kv_elem_bytes=spec.cache_elem_bytes)
    kv_bytes_step = bytes_layer.kv * spec.num_layers
    for _ in range(max(3, warmup)):
        step.run()
    torch.cuda.synchronize()
    st, flags = pkv.device_status(dev)
    if st != 0:
        raise RuntimeError(f"{spec.name}: device status {st} flags {flags:#x} after warm-up")

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step.run()
        for _ in range(max(3, warmup)):
            graph.replay()
    torch.cuda.synchronize()

    flush = kv_bytes_step < 4 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def region():
        if flush:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(steps)]
            with torch.cuda.stream(stream):
                for a0, a1 in pairs:
                    scrub.fill_(1)
                    a0.record(stream)
                    graph.replay()
                    a1.record(stream)
            torch.cuda.synchronize()
            return sum(a0.elapsed_time(a1) for a0, a1 in pairs)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    with ClockSampler(torch.cuda.current_device()) as clocks:
        regions = timed_regions(region, min_ms, world, dev)
    clock = clocks.summary()
    ms_total = sum(regions)
    n_steps = steps * len(regions)
    ms_step = ms_total / n_steps
    st, flags = pkv.device_status(dev)
    if st != 0:
        raise RuntimeError(f"{spec.name}: device status {st} flags {flags:#x} after the timed region")

    # Dominant kernel.  When the step is that kernel alone (fused step, merge
    # in the kernel) its mean launch duration over the timed region is the
    # step time over the launches; otherwise the attention call is timed per
    # launch with events on its stream, eager, over a few steps.
    n_steps_ev = 3
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(spec.num_layers)] for _ in range(n_steps_ev)]
    torch.cuda.synchronize()
    for i in range(n_steps_ev):
        step.run(events=evs[i])
    torch.cuda.synchronize()
    eager_ms = statistics.mean(a.elapsed_time(b) for e in evs for a, b in e)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    launch_bytes = bytes_layer.attention + (bytes_layer.append if step.fused else 0)
    only_dominant = step.fused and not opts.get("separate_reduce")
    launch_ms = ms_step / spec.num_layers if only_dominant else eager_ms
    achieved = launch_bytes / (launch_ms * 1e-3) / 1e9
    kernel_name = decode_kernel_name(spec, kernel, step.fused)
    kv_total = sum_over_ranks(kv_bytes_step, world, dev)
    value = kv_total / (ms_step * 1e-3) / 1e9
    res = {
        "value": round(value, 1), "unit": UNIT, "ms_per_step": round(ms_step, 4),
        "decode_tokens_per_s": round(sum_over_ranks(B, world, dev) / (ms_step * 1e-3), 1),
        "frac_of_measured_hbm": round(value / world / peak, 4),
        "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "dtype": spec.cache_dtype, "q_dtype": spec.dtype,
        "workload": f"{spec.name}: {spec.num_layers} layers x {B} seqs, ctx {int(pl.context_lens.min())}.."
                    f"{int(pl.context_lens.max())} (sum {int(pl.context_lens.sum())}, appended token included), "
                    f"{spec.num_q_heads}q/{spec.num_kv_heads}kv heads, D{spec.head_dim}, {spec.dtype}"
                    + (f" q, {spec.cache_dtype} cache (scales {spec.kv_scales[0]:.6g}, {spec.kv_scales[1]:.6g})"
                       if spec.fp8 else "") + f", block {spec.block_size}, {pl.num_blocks}-block pool",
        "kv_bytes_per_step": kv_bytes_step,
        "timed": {"regions": len(regions), "steps_per_region": steps, "steps": n_steps,
                  "ms": round(ms_total, 3)},
        "l2": ("L2 flushed (a %d MB write) before each timed replay: the step reads %.3f GB of K/V"
               % (2 * L2_BYTES // 10**6, kv_bytes_step / 1e9)) if flush else
              "no flush: each step reads %.2f GB of K/V (> 4x the 129 MB L2)" % (kv_bytes_step / 1e9),
        "timing": ("CUDA-graph replay of the whole step (%d launches), CUDA events on the replay stream"
                   % step.launches_per_step),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(kernel_name, spec.name),
                     "kernel": kernel_name + (" + paged_decode_reduce_kernel" if opts.get("separate_reduce")
                                              else " (cross-CTA merge fused)"),
                     "algorithmic_bytes_per_launch": launch_bytes,
                     "launch_ms": round(launch_ms, 5),
                     "launch_ms_source": ("timed graph replays / launches (the step is only this kernel)"
                                          if only_dominant else "eager CUDA events around each call"),
                     "eager_launch_ms": round(eager_ms, 5), "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clock,
    }
    if spec.prefix_tokens:
        uniq = pl.unique_kv_tokens * spec.num_kv_heads * spec.head_dim * 2 * spec.cache_elem_bytes
        res["unique_kv_bytes_per_step"] = uniq * spec.num_layers
        res["unique_kv_gbs"] = round(sum_over_ranks(uniq * spec.num_layers, world, dev) / (ms_step * 1e-3) / 1e9, 1)
        res["note"] = ("value counts every sequence's K/V (the logical bytes the method reads); "
                       "unique_kv_gbs counts each shared prefix block once")
    res["_launches_per_step"] = step.launches_per_step
    del graph
    return res, step


def e2e_measure(step, args, world, dev):
    """The same step through the public API with host buffers: the step's
    inputs copied from pinned host memory and its outputs copied back, inside
    the timed region."""
    pl = step.pl
    h_q = step.q.cpu().pin_memory()
    h_kn = step.kn.cpu().pin_memory()
    h_vn = step.vn.cpu().pin_memory()
    h_tab = torch.from_numpy(pl.block_tables).pin_memory()
    h_ctx = torch.from_numpy(pl.context_lens).pin_memory()
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_tab, h_ctx))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        step.q.copy_(h_q, non_blocking=True)
        step.kn.copy_(h_kn, non_blocking=True)
        step.vn.copy_(h_vn, non_blocking=True)
        step.tables.copy_(h_tab, non_blocking=True)
        step.ctx.copy_(h_ctx, non_blocking=True)
        step.run()
        h_out.copy_(step.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.e2e_steps):
        e2e_step()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.e2e_steps
    return e2e_ms, h2d, d2h


def bench_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, True)
    spec = SPECS[args.workload]
    if args.layers:
        spec = dataclasses.replace(spec, num_layers=args.layers)
    opts = decode_opts(args)
    res, step = measure_decode(spec, args, dev, world, args.min_timed_ms, args.steps, args.warmup,
                               kernel=args.kernel, fused=not args.unfused, opts=opts)
    launches = res.pop("_launches_per_step")
    e2e_ms, h2d, d2h = e2e_measure(step, args, world, dev)
    kv_total = sum_over_ranks(res["kv_bytes_per_step"], world, dev)
    pl, B = step.pl, step.B
    result = {
        "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.cache_dtype, "accumulate": "f32",
        "q_dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, random block placement)",
        "config": {"workload": f"{spec.name}: {spec.num_layers} layers x {B} seqs x "
                               f"{int(pl.context_lens.max())} ctx (appended token included), "
                               f"{spec.num_q_heads}q/{spec.num_kv_heads}kv heads, D{spec.head_dim}, "
                               f"{spec.dtype}" + (f" q, {spec.cache_dtype} cache (scales "
                                                  f"{spec.kv_scales[0]:.6g}, {spec.kv_scales[1]:.6g})"
                                                  if spec.fp8 else "") +
                               f", block {spec.block_size}, {pl.num_blocks}-block pool",
                   "num_layers": spec.num_layers, "num_seqs": B, "context_tokens": int(pl.context_lens.sum()),
                   "kv_bytes_per_step": res["kv_bytes_per_step"], "kernel": args.kernel,
                   "timing": res["timing"] + "; regions of exactly --steps replays repeated until "
                             f"{args.min_timed_ms:.0f} ms of device time",
                   "l2": res["l2"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "timed": res["timed"],
        "decode_tokens_per_s": res["decode_tokens_per_s"],
        "frac_of_nominal_8tbs": res["frac_of_nominal_8tbs"],
        "frac_of_measured_hbm": res["frac_of_measured_hbm"],
        "e2e": {"value": round(kv_total / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "python binding -> C ABI, pinned host buffers, copies in the timed region"},
        "gpu_launches": launches * res["timed"]["steps"],
        "roofline": res["roofline"],
        "clocks": res["clocks"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(spec, pl, args.cpu_seconds, step, args.cpu_single_seconds)
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    names = []
    if args.configs != "none":
        names = list(CONFIG_ORDER) if args.configs == "all" else [n.strip() for n in args.configs.split(",")]
    configs = {}
    for name in names:
        if name == spec.name:
            continue
        try:
            configs[name] = measure_config(name, args, dev, world, rank, local)
        except Exception as exc:  # one failing entry must not hide the others
            configs[name] = {"error": f"{type(exc).__name__}: {exc}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if configs:
        result["configs"] = configs
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_config(name, args, dev, world, rank, local):
    """One entry of `configs`: the workload's step timed like the headline."""
    if name == "swap":
        line = bench_swap(args, world, rank, local, emit=False)
        keep = ("value", "unit", "swap_out_gbs", "swap_in_gbs", "copy_engine_d2h_gbs", "copy_engine_h2d_gbs",
                "page_request_out_and_back_ms", "round_trip_exact", "timed", "clocks", "config")
        return {k: line[k] for k in keep if k in line}
    spec = SPECS[name]
    if spec.new_tokens:
        line = bench_prefill(args, world, rank, local, spec_name=name, emit=False)
        keep = ("value", "unit", "ms_per_step", "attention_ms_per_layer", "attention_tflops",
                "kv_gbs_per_layer", "roofline", "timed", "clocks", "config")
        return {k: line[k] for k in keep if k in line}
    min_ms = args.config_min_timed_ms
    res, step = measure_decode(spec, args, dev, world, min_ms, max(3, min(args.steps, 20)), args.warmup,
                               kernel="auto", fused=True, opts=dict(pdl=True, early_reads=True))
    res.pop("_launches_per_step")
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if spec.num_layers == 1 and "flushed" in res["l2"]:
        # The same launch rotated over independent layer pools, back to back
        # in one graph: each launch reads a pool the others evicted from L2.
        spec_r = dataclasses.replace(spec, num_layers=BACK_TO_BACK_POOLS)
        rot, step = measure_decode(spec_r, args, dev, world, min_ms, max(3, min(args.steps, 20)),
                                   args.warmup, kernel="auto", fused=True, opts=dict(pdl=True, early_reads=True))
        del step
        res["back_to_back"] = {
            "what": f"{BACK_TO_BACK_POOLS} independent pools of this layer back to back in one graph "
                    f"({rot['kv_bytes_per_step'] / 1e9:.2f} GB per replay, no flush)",
            "value": rot["value"], "ms_per_launch": round(rot["ms_per_step"] / BACK_TO_BACK_POOLS, 5),
            "roofline_frac": rot["roofline"]["frac"], "clocks": rot["clocks"]}
    return res


# ------------------------------------------------------------- oracle arm
def oracle_sample(spec, pl, layer_pools=None, device="cpu"):
    """Host inputs of one layer's sampled step for the oracle (compact pool)."""
    if layer_pools is None:
        kc, vc = pool_layer_values(spec, pl.num_blocks, 0, device)
    else:
        kc, vc = layer_pools
    rows = pl.block_tables
    used = np.unique(rows[rows >= 0])
    remap = np.full(pl.num_blocks, -1, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    tabs = np.where(rows >= 0, remap[np.maximum(rows, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).to(kc.device)
    if kc.element_size() == 1:  # E4M3: gather through byte views
        return (kc.view(torch.uint8)[idx].cpu().view(kc.dtype), vc.view(torch.uint8)[idx].cpu().view(vc.dtype),
                tabs)
    return kc[idx].cpu(), vc[idx].cpu(), tabs


def _oracle_rate(spec, pl, q, kc, vc, tabs, seconds, nthreads):
    """KV bytes per second of the oracle over whole sequences of layer 0, one
    sequence at a time until `seconds` have passed (at least one)."""
    import oracle

    B = len(pl.context_lens)
    scales = dict(k_scale=spec.kv_scales[0], v_scale=spec.kv_scales[1]) if spec.fp8 else {}
    t0 = time.perf_counter()
    done_bytes = 0
    n = 0
    while True:
        s = n % B
        oracle.paged_decode(q[s:s + 1], kc, vc, tabs[s:s + 1], pl.context_lens[s:s + 1], spec.attn_scale,
                            nthreads=nthreads, **scales)
        done_bytes += int(pl.context_lens[s]) * spec.num_kv_heads * spec.head_dim * 2 * spec.cache_elem_bytes
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return done_bytes / dt / 1e9, n, done_bytes, dt


def cpu_baseline(spec, pl, seconds, step=None, single_seconds=4.0):
    """The oracle (as it stands) on layer 0 of the workload: all host cores for
    ~`seconds`, then one thread for ~`single_seconds`."""
    import oracle
    from paged_kv_cache_slots_gb300 import roofline

    B = len(pl.context_lens)
    if step is not None:
        kc, vc, tabs = oracle_sample(spec, pl, step.layers[0])
        q = step.q[0].cpu()
    else:
        kc, vc, tabs = oracle_sample(spec, pl)
        q, _, _ = step_layer_values(spec, B, 0, "cpu")
    cores = oracle.num_cores()
    b = roofline.attention_bytes(pl.context_lens, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                 spec.elem_bytes, spec.block_size, spec.elem_bytes, 0,
                                 kv_elem_bytes=spec.cache_elem_bytes)
    rate, n, done, dt = _oracle_rate(spec, pl, q, kc, vc, tabs, seconds, cores)
    out = {"value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"layer 0, {n} sequence passes (all {spec.num_q_heads} query heads each), "
                     f"{done / 1e9:.2f} GB of K/V in {dt:.1f} s",
           "full_layer_kv_bytes": b.kv}
    if single_seconds > 0:
        rate1, n1, done1, dt1 = _oracle_rate(spec, pl, q, kc, vc, tabs, single_seconds, 1)
        out["single_thread"] = {"value": round(rate1, 4), "unit": UNIT, "cores": 1,
                                "sample": f"layer 0, {n1} sequence passes, {done1 / 1e9:.3f} GB of K/V "
                                          f"in {dt1:.1f} s"}
    return out


def bench_reference(args, world, rank):
    """The oracle as the reference arm: host cores, bounded samples of the workload."""
    import oracle

    if rank != 0:
        return
    spec = SPECS[args.workload]
    pl = make_placement(spec)
    kc, vc, tabs = oracle_sample(spec, pl)
    B = len(pl.context_lens)
    q, _, _ = step_layer_values(spec, B, 0, "cpu")
    cores = oracle.num_cores()

    scales = dict(k_scale=spec.kv_scales[0], v_scale=spec.kv_scales[1]) if spec.fp8 else {}

    def one(i):
        s = i % B
        oracle.paged_decode(q[s:s + 1], kc, vc, tabs[s:s + 1], pl.context_lens[s:s + 1], spec.attn_scale,
                            nthreads=cores, **scales)
        return int(pl.context_lens[s]) * spec.num_kv_heads * spec.head_dim * 2 * spec.cache_elem_bytes

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    done = sum(one(i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/K/V, random block placement)",
        "config": {"workload": f"{spec.name} (oracle arm: each step is one sequence of layer 0, "
                               f"all {spec.num_q_heads} query heads)"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x one sequence of layer 0 of {spec.name}"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------- prefill leg
def bench_prefill(args, world, rank, local, spec_name=None, emit=True):
    """A multi-token step (chunked prefill next to decodes): for every layer
    the varlen slot mapping, the append of every new token and the causal
    attention of the new tokens over the paged cache, captured in a CUDA graph.
    value = new tokens per second; the roofline is the attention's causal
    FLOPs (4 * D * Hq per (query, visible key) pair) against the bf16 tensor
    peak (the sustained rate: the kernel runs inside a step of ~0.27 s)."""
    import paged_kv_cache_slots_gb300 as pkv
    from workloads import step_token_values
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, True)
    name = spec_name or (args.workload if SPECS[args.workload].new_tokens else "chunked_prefill_b32")
    spec = SPECS[name]
    if args.layers and spec_name is None:
        spec = dataclasses.replace(spec, num_layers=args.layers)
    if args.block_size and spec_name is None:
        spec = dataclasses.replace(spec, block_size=args.block_size)
    pl = make_placement(spec)
    ctx = pl.context_lens
    nq = np.asarray(spec.new_tokens, np.int32)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    T = int(qs[-1])
    pool = pkv.KVPool(spec.num_layers, pl.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim,
                      spec.torch_dtype, device=device)
    layers = [pool.layer(l) for l in range(spec.num_layers)]
    for l, (kc, vc) in enumerate(layers):
        fill_pool_layer(spec, l, kc, vc)
    qkv = [step_token_values(spec, T, l, device) for l in range(spec.num_layers)]
    tables = torch.from_numpy(pl.block_tables).to(device)
    ctx_d = torch.from_numpy(ctx).to(device)
    qs_d = torch.from_numpy(qs).to(device)
    slots = torch.empty(T, dtype=torch.int32, device=device)
    out = torch.empty((T, spec.num_q_heads, spec.head_dim), dtype=spec.torch_dtype, device=device)
    ws = torch.empty(int(pkv.load_library().paged_prefill_workspace_bytes(len(ctx))), dtype=torch.uint8,
                     device=device)

    def step():
        pkv.slot_mapping_varlen(tables, qs_d, ctx_d, spec.block_size, pl.num_blocks, num_tokens=T, out=slots)
        for l, (kc, vc) in enumerate(layers):
            q, kn, vn = qkv[l]
            pool.append(l, kn, vn, slots)
            pkv.paged_prefill_attention(q, kc, vc, tables, qs_d, ctx_d, spec.attn_scale, out=out, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, flags = pkv.device_status(device)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x} after warm-up")
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream(device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
        graph.replay()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 3 if spec_name else 20))

    def region():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    min_ms = args.config_min_timed_ms if spec_name else args.min_timed_ms
    with ClockSampler(local) as clocks:
        regions = timed_regions(region, min_ms, world, device)
    ms_step = sum(regions) / (steps * len(regions))
    # Attention alone, one layer, events on its stream (the dominant kernel).
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(6)]
    for a, b in ev:
        a.record()
        pkv.paged_prefill_attention(qkv[0][0], layers[0][0], layers[0][1], tables, qs_d, ctx_d, spec.attn_scale,
                                    out=out, workspace=ws)
        b.record()
    torch.cuda.synchronize()
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[1:])
    visible = sum(int(n) * (int(c) - int(n)) + int(n) * (int(n) + 1) // 2 for n, c in zip(nq, ctx))
    # The library takes the tcgen05 kernel for head_dim 128 and blocks that tile 64 keys.
    tc = spec.head_dim == 128 and (spec.block_size % 64 == 0 or 64 % spec.block_size == 0)
    kernel_name = ("paged_prefill_tc_kernel<%s,G%d,bs%d>" % (spec.dtype, spec.num_q_heads // spec.num_kv_heads,
                                                             spec.block_size)
                   if tc else "paged_prefill_kernel<%s,%d>" % (spec.dtype, spec.head_dim))
    flops_layer = 4.0 * spec.head_dim * spec.num_q_heads * visible
    peaks, peak_kind = measured_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
    peak_burst = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops_layer / (attn_ms * 1e-3) / 1e12
    kv_layer = int(ctx.sum()) * spec.num_kv_heads * spec.head_dim * 2 * spec.elem_bytes
    line = {
        "metric": "chunked-prefill step new tokens/s",
        "value": round(T * world / (ms_step * 1e-3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, random block placement)",
        "config": {"workload": f"{spec.name}: {spec.num_layers} layers, {len(ctx)} sequences, {T} new tokens "
                               f"({int((nq == 1).sum())} decodes + chunks {sorted(int(n) for n in nq if n > 1)}), "
                               f"contexts up to {int(ctx.max())}, 32q/8kv heads, D{spec.head_dim}, "
                               f"block {spec.block_size}, {pl.num_blocks}-block pool",
                   "timing": "CUDA-graph replay of the whole step, CUDA events on the replay stream",
                   "l2": "each layer reads %.2f GB of K/V (> 129 MB L2)" % (kv_layer / 1e9)},
        "timed": {"regions": len(regions), "steps_per_region": steps, "steps": steps * len(regions),
                  "ms": round(sum(regions), 3)},
        "attention_ms_per_layer": round(attn_ms, 4),
        "attention_tflops": round(achieved, 1),
        "kv_gbs_per_layer": round(kv_layer / (attn_ms * 1e-3) / 1e9, 1),
        "gpu_launches": steps * len(regions) * (1 + 3 * spec.num_layers),  # slots; append, plan, attention a layer
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tf, 4), "frac_of_burst": round(achieved / peak_burst, 4),
                     "traffic": recorded_traffic(kernel_name, spec.name, PREFILL_SOURCES),
                     "kernel": kernel_name + " (one layer, eager, CUDA events)",
                     "algorithmic_flops_per_launch": flops_layer,
                     "peak_source": f"{peak_kind} bf16_tflops_sustained (cuBLAS, seconds-long loop)"},
        "clocks": clocks.summary(),
    }
    del graph, pool, layers, qkv
    if emit and rank == 0:
        print(json.dumps(line), flush=True)
    return line


# ------------------------------------------------------------- swap leg
def bench_swap(args, world, rank, local, emit=True):
    """Swap-out and swap-in throughput of whole KV blocks (every layer's K and V)
    between the pool and page-locked host memory, for the preempted request of
    "Batching and Scheduling", Example 8: 2000 tokens of the 8B shape (125
    blocks of 16 tokens, 32 layers, 8 KV heads, head_dim 128, bf16), i.e.
    250 MiB each way, `--swap-requests` such requests per copy.  The link's
    own ceiling is measured beside it: one contiguous cudaMemcpyAsync of the
    same byte count each way through the copy engines."""
    import paged_kv_cache_slots_gb300 as pkv
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, True)
    per_req = 125
    nreq = max(1, args.swap_requests)
    nblk = per_req * nreq
    pool = pkv.KVPool(32, 2 * nblk + 16, 16, 8, 128, torch.bfloat16, device=device)
    pool.buffer.view(torch.int16).random_(generator=torch.Generator(device=device).manual_seed(5))
    perm = torch.randperm(2 * nblk + 16, generator=torch.Generator().manual_seed(9))
    ids = perm[:nblk].to(torch.int32).to(device)
    nbytes = pool.swap_bytes(nblk)
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev_copy = torch.empty(nbytes, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    reps = max(1, min(args.steps, 50))
    min_ms = args.config_min_timed_ms if not emit else 0.0
    total_reps = [0]

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()

        def region():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        regions = timed_regions(region, min_ms, world, device)
        total_reps[0] += reps * len(regions)
        return sum(regions) / (reps * len(regions))

    with ClockSampler(local) as clocks:
        out_ms = timed(lambda: pool.swap_out(ids, host=host))
        in_ms = timed(lambda: pool.swap_in(ids, host))
        ce_out_ms = timed(lambda: host.copy_(dev_copy, non_blocking=True))
        ce_in_ms = timed(lambda: dev_copy.copy_(host, non_blocking=True))
    # The copies above are checked, not only timed: the pool must round-trip.
    before = pool.buffer.clone()
    pool.swap_out(ids, host=host)
    for layer in (0, 31):
        for t in pool.layer(layer):
            t[ids.long()] = 0
    pool.swap_in(ids, host)
    torch.cuda.synchronize()
    blocks_ok = bool(torch.equal(pool.buffer, before))
    status, flags = pkv.device_status(device)
    gbs = lambda ms: nbytes * world / (ms * 1e-3) / 1e9  # noqa: E731
    page_bytes = pool.swap_bytes(per_req)
    line = {
        "metric": "KV swap GB/s (host memory, out and back)",
        "value": round(2 * nbytes * world / ((out_ms + in_ms) * 1e-3) / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": reps,
        "warmup": max(3, args.warmup),
        "higher_is_better": True,
        "scaling": "weak",
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"swap {nreq} x 2000-token 8B-shaped requests "
                               f"({nblk} blocks, {nbytes / 2**20:.0f} MiB each way)",
                   "host_memory": "page-locked", "l2": "inputs larger than L2"},
        "swap_out_gbs": round(gbs(out_ms), 1),
        "swap_in_gbs": round(gbs(in_ms), 1),
        "copy_engine_d2h_gbs": round(gbs(ce_out_ms), 1),
        "copy_engine_h2d_gbs": round(gbs(ce_in_ms), 1),
        "page_request_out_and_back_ms": round((out_ms + in_ms) * page_bytes / nbytes, 3),
        "page_request_pcie4_ms": round(2 * page_bytes / 31.5e9 * 1e3, 1),
        "round_trip_exact": blocks_ok,
        "device_status": [status, flags],
        "timed": {"copies": total_reps[0]},
        "gpu_launches": 2 * reps,
        "clocks": clocks.summary(),
        "vs_baseline": None,
    }
    del pool, host, dev_copy, before
    if emit and rank == 0:
        print(json.dumps(line), flush=True)
    return line


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        bench_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    if args.swap:
        bench_swap(args, world, rank, local)
        return
    if args.prefill or SPECS[args.workload].new_tokens:
        bench_prefill(args, world, rank, local)
        return
    bench_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
