#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

One step = one fused attention forward over the whole workload (default: the
Llama-2-7B-shaped causal prefill, B=4, S=2048, Hq=Hkv=32, D=128, bf16) with
inputs resident in device memory. Prints ONE JSON line on rank 0.

  value      TFLOP/s = 4*B*Hq*Sq*Sk*D (halved for causal) per step x steps x
             ranks / max-over-ranks device time (CUDA events around each launch,
             L2 flushed by an untimed 256 MiB write before every step)
  e2e        the same metric through the public host-buffer call (attn_fwd_host)
             with pinned host Q/K/V/O/LSE: every step copies its inputs in and
             its outputs back, pipelined with the computation, all inside the
             timed region
  roofline   the kernel against the measured dense bf16 tensor peak
  cpu_baseline  the FP64 oracle on this host's cores, on a bounded sample
  configs    the other causal D=128 prefills (GQA B8 S4096 and long-context GQA
             B1 S16384 by default), each timed the same way: value, roofline,
             median and min launch time, clocks

`--rope` runs the same workload with the rotary position embedding: each step
rotates the keys once (bandwidth-bound pass) and runs the attention kernel that
rotates the queries at tile load; `value` covers both launches, `roofline` the
attention kernel alone, and the FLOP count stays the attention's.
`--block` runs the attention block of one Llama-2-7B-sized layer (LayerNorm,
QKV projection, attention, output projection and residual; B=4, S=2048,
hidden 4096) as its four kernels with CUDA events between them: `value` is the
block's algorithmic TFLOP/s (both projections plus the causal attention),
`roofline` the QKV projection GEMM, its dominant kernel.
`--decode [--decode-config NAME]` times the split-key path on a decode workload
(one new query row per sequence over a KV cache): `value` is the algorithmic
bytes (Q, K, V read once, O and LSE written once) per second, the roofline HBM.
`--impl reference` times the oracle (the only reference implementation this
method has) on the same workload and metric instead.
Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU (the forward shards over (b, head) with no exchange), so the scaling
is weak; the barrier and max-over-ranks timing are host-side plumbing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from transformer_attention_02_gb300 import inputs as I  # noqa: E402

METRIC = "fused attention fwd TFLOP/s (bf16) and % of GB300 dense bf16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# Sources that decide each profiled kernel's code (the profile summaries record their hash).
KERNEL_SOURCES = {
    "attention": ["transformer_attention_02_gb300/csrc/" + f for f in (
        "attn_kernel.cuh", "ptx.cuh", "attn_api.cu", "attn_launch.h", "attn_fwd_inst.cuh", "fwd_bf16.cu",
        "fwd_f16.cu", "fwd_rope_bf16.cu", "fwd_rope_f16.cu", "fwd_pack_bf16.cu", "fwd_pack_f16.cu")],
    "gemm": ["transformer_attention_02_gb300/csrc/" + f for f in (
        "gemm_kernel.cuh", "block_params.h", "block_kernels.cu", "attn_kernel.cuh", "ptx.cuh", "attn_api.cu")],
}
ROPE_BASE = 10000.0


# ------------------------------------------------------------------ helpers

def kernel_source_hash(kernel: str = "attention") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(summary: str, kernel: str = "attention"):
    """DRAM bytes per launch from the committed ncu summary profiles/<summary>.md,
    if it was taken on the current sources of that kernel (same hash); otherwise None."""
    path = os.path.join(ROOT, "profiles", f"{summary}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for t, s in self.samples if t0 <= t <= t1]
        if not rows:      # window shorter than the sampling period: nearest samples
            rows = [s for t, s in sorted(self.samples, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))[:3]]
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, device) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_tflops(flops_per_step: float, steps: int, n_ranks: int, max_seconds: float) -> float:
    return flops_per_step * steps * n_ranks / max_seconds / 1e12


# ----------------------------------------------------------- CPU oracle arm

def row_flops(cfg: I.AttnConfig, r0: int, r1: int) -> float:
    """Algorithmic FLOPs of query rows [r0, r1) of one (b, h) slice."""
    tot = 0.0
    for i in range(r0, r1):
        vis = min(cfg.Sk, max(0, i + cfg.Sk - cfg.Sq + 1)) if cfg.causal else cfg.Sk
        tot += 4.0 * cfg.D * vis
    return tot


def oracle_sample(cfg, q, k, v, mask, target_s: float, slices_cycle, rope_kw=None):
    """Time the oracle on whole (b, h) slices until about target_s seconds of
    work are done (at least one slice). Returns (seconds, flops, n_slices, threads)."""
    import oracle
    orc = oracle.Oracle()
    qb, kb, vb = I.bits(q), I.bits(k), I.bits(v)
    mk = None if mask is None else mask.numpy()
    per_slice = row_flops(cfg, 0, cfg.Sq)
    done, spent, n = 0.0, 0.0, 0
    while n == 0 or (spent < target_s and n < len(slices_cycle)):
        t0 = time.perf_counter()
        orc.attention(qb, kb, vb, mask_kind=cfg.mask_kind, mask=mk, slices=[slices_cycle[n]],
                      **(rope_kw or {}))
        spent += time.perf_counter() - t0
        done += per_slice
        n += 1
    return spent, done, n, orc.num_threads()


def spread_slices(cfg):
    """(b, h) slices spread over the batch and heads (deterministic order)."""
    out, seen = [], set()
    total = cfg.B * cfg.Hq
    step = max(1, total // 64)
    for idx in list(range(0, total, step)) + list(range(total)):
        s = (idx // cfg.Hq, idx % cfg.Hq)
        if s not in seen:
            seen.add(s)
            out.append(s)
    return out


def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v, mask = I.make_inputs(cfg)
    import oracle
    orc = oracle.Oracle()
    qb, kb, vb = I.bits(q), I.bits(k), I.bits(v)
    mk = None if mask is None else mask.numpy()
    slices = spread_slices(cfg)
    rope_kw = dict(rope_base=ROPE_BASE, rope_round=True) if args.rope else {}
    # size each step (a window of query rows of one slice) so the whole run takes about a minute
    budget = 60.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    orc.attention(qb, kb, vb, mask_kind=cfg.mask_kind, mask=mk, slices=[slices[0]], rows=(0, 16), **rope_kw)
    per_row = max(1e-6, (time.perf_counter() - t0) / 16)
    rows = int(max(8, min(cfg.Sq, budget / per_row / 1.5)))

    def step(i):
        b, h = slices[i % len(slices)]
        r0 = (i * 977 * rows) % max(1, cfg.Sq - rows + 1)
        orc.attention(qb, kb, vb, mask_kind=cfg.mask_kind, mask=mk, slices=[(b, h)], rows=(r0, r0 + rows),
                      **rope_kw)
        return row_flops(cfg, r0, r0 + rows)

    for i in range(args.warmup):
        step(i)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += step(args.warmup + i)
    sec = time.perf_counter() - t0
    value = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_json(cfg, args.rope),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                         "sample": f"{args.steps} steps of {rows} query rows of one (b,h) slice each, "
                                   f"slices spread over the batch and heads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def config_json(cfg, rope=False):
    extra = {"rope": {"base": ROPE_BASE, "q_pos0": 0, "k_pos0": 0, "pairs": "interleaved"}} if rope else {}
    return {**extra, "workload": cfg.name + ("+rope" if rope else ""), "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
            "Sq": cfg.Sq, "Sk": cfg.Sk,
            "D": cfg.D, "mask": ("causal" if cfg.causal else "none") + ("+additive" if cfg.additive_mask else ""),
            "values": cfg.values, "seed": cfg.seed,
            "l2": "flushed before every timed step (untimed 256 MiB write); device time = CUDA events "
                  "around each launch"}


def time_config(A, cfg, steps, warmup, dev, stream, flush, clocks, world, peak, peak_src):
    """Device time of `steps` launches of the fused attention on one more workload,
    measured like the headline (inputs resident, L2 flushed before each launch,
    CUDA events around each launch, max over ranks)."""
    q, k, v, mask = I.make_inputs(cfg)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if mask is None else mask.to(dev)
    del q, k, v, mask
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), dtype=torch.float32, device=dev)

    def launch():
        A.attention(qd, kd, vd, causal=cfg.causal, mask=md, out=o, lse=lse, stream=stream)

    for _ in range(warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize(dev)
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError(f"kernel reported a device timeout during warm-up ({cfg.name})")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError(f"kernel reported a device timeout in the timed region ({cfg.name})")
    ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    max_s = reduce_max(sum(ms) / 1e3, dev)
    achieved = cfg.flops / (sum(ms) / 1e3 / steps) / 1e12
    return {
        "value": whole_job_tflops(cfg.flops, steps, world, max_s), "unit": UNIT, "steps": steps, "warmup": warmup,
        "ms_per_step": max_s / steps * 1e3, "config": config_json(cfg),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": profiled_traffic("attn_fwd_" + cfg.name),
                     "peak_source": f"{peak_src} bf16_tflops (burst, kernel timed alone)",
                     "kernel": "attn_fwd_kernel", "median_ms": statistics.median(ms), "min_ms": min(ms)},
        "clocks": clocks.summary(t0, t1),
        "gpu_launches": steps,
    }


def run_ours(args, cfg):
    import torch.distributed as dist
    from transformer_attention_02_gb300 import attn as A

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    A.lib()

    q, k, v, mask = I.make_inputs(cfg)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if mask is None else mask.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.rope:
        table = A.rope_table(max(cfg.Sq, cfg.Sk), cfg.D, ROPE_BASE, stream=stream)
        k_rot = torch.empty_like(kd)

    def launch_keys():          # rotary variant only: rotate each key once
        A.rope_apply(kd, table, pos0=0, out=k_rot, stream=stream)

    def launch_attention():
        if args.rope:
            A.attention_rope(qd, k_rot, vd, table, k_rot=None, causal=cfg.causal, mask=md, out=o, lse=lse,
                             stream=stream)
        else:
            A.attention(qd, kd, vd, causal=cfg.causal, mask=md, out=o, lse=lse, stream=stream)

    def launch():
        if args.rope:
            launch_keys()
        launch_attention()

    for _ in range(args.warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize(dev)
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError("kernel reported a device timeout during warm-up")

    clocks = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        if args.rope:
            launch_keys()
        mids[i].record(stream)
        launch_attention()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_ms = [m.elapsed_time(e) for m, e in zip(mids, ends)]      # the attention kernel alone
    key_ms = [s.elapsed_time(m) for s, m in zip(starts, mids)] if args.rope else None
    local_s = sum(step_ms) / 1e3
    max_s = reduce_max(local_s, dev)
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError("kernel reported a device timeout in the timed region")

    # ---- end to end through the public API with pinned host buffers
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    mh = None if mask is None else mask.pin_memory()
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))

    host_ws = None
    if not args.rope:
        host_ws = torch.empty(max(1, A.attn_fwd_host_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, cfg.D,
                                                                       cfg.mask_kind)), dtype=torch.uint8, device=dev)

    def e2e_step():
        if not args.rope:
            # the public host-buffer call: pipelined copies in, compute, copies out
            A.attention_host(qh, kh, vh, causal=cfg.causal, mask=mh, out=oh, lse=lh, workspace=host_ws,
                             device=dev, stream=stream)
            return
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        if mh is not None:
            md.copy_(mh, non_blocking=True)
        launch()
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3, dev)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh)) + (0 if mh is None else mh.numel() * 4)
    d2h = oh.numel() * oh.element_size() + lh.numel() * 4

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # The other causal D=128 prefills, measured the same way on the same GPU.
    extra = {}
    names = [n for n in (args.extra_configs.split(",") if args.extra_configs else []) if n and n != cfg.name]
    if names and not args.rope:
        del qd, kd, vd, o, lse, md
        torch.cuda.empty_cache()
        for name in names:
            extra[name] = time_config(A, I.CONFIGS[name], max(3, min(args.steps, 200)), args.warmup, dev, stream,
                                      flush, clocks, world, peak, peak_src)
            torch.cuda.empty_cache()

    if rank == 0:
        clocks.stop()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    flops = cfg.flops
    value = whole_job_tflops(flops, args.steps, world, max_s)
    per_launch_s = sum(kernel_ms) / 1e3 / args.steps
    achieved = flops / per_launch_s / 1e12
    traffic = profiled_traffic("attn_fwd_" + cfg.name + ("_rope" if args.rope else ""))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_json(cfg, args.rope),
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst, kernel timed alone)",
                     "kernel": "attn_fwd_kernel", "median_ms": statistics.median(kernel_ms),
                     "min_ms": min(kernel_ms)},
        "e2e": {"value": whole_job_tflops(flops, e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "attention_rope + explicit copies" if args.rope else
                       "attention_host (attn_fwd_host: pipelined host-buffer call)"},
        "gpu_launches": args.steps * (2 if args.rope else 1) + sum(e["gpu_launches"] for e in extra.values()),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "wall_s_timed_region": t_wall1 - t_wall0,
        "kernel_source_hash": kernel_source_hash(),
    }
    if cfg.additive_mask:
        # The tensor roofline is the nominal one; what the masked kernel actually
        # hits (ncu) is the L1 throughput of the FP32 mask rows, one row per
        # thread.
        line["roofline"]["limiter"] = "L1 throughput of the FP32 mask-row loads (32 rows per warp request)"
    if extra:
        line["configs"] = extra
    if args.rope:
        kv_bytes = 2 * cfg.B * cfg.Sk * cfg.Hkv * cfg.D * 2          # read K, write rotated K
        med = statistics.median(key_ms)
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        line["key_rotation"] = {"kernel": "rope_apply_kernel", "median_ms": med, "bytes": kv_bytes,
                                "achieved_gbs": kv_bytes / (med / 1e3) / 1e9, "peak_gbs": hbm,
                                "frac": kv_bytes / (med / 1e3) / 1e9 / hbm,
                                "share_of_step": sum(key_ms) / sum(step_ms)}
    if world == 1 and not args.no_cpu_baseline:
        rope_kw = dict(rope_base=ROPE_BASE, rope_round=True) if args.rope else None
        sec, done, n, threads = oracle_sample(cfg, q, k, v, mask, args.cpu_seconds, spread_slices(cfg), rope_kw)
        line["cpu_baseline"] = {"value": done / sec / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n} of {cfg.B * cfg.Hq} (b,h) slices, all rows, "
                                          f"{sec:.1f} s of FP64 oracle time"}
    print(json.dumps(line), flush=True)
    return 0


def run_block(args):
    """The attention block, one step = LayerNorm -> QKV GEMM -> attention -> output GEMM (+ residual)."""
    import torch.distributed as dist
    from transformer_attention_02_gb300 import attn as A

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    A.lib()
    cfg = I.BLOCK_CONFIGS["llama2_7b_block"]
    host = I.make_block_inputs(cfg)
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o = (t.to(dev) for t in host)
    M, H, F = cfg.B * cfg.S, cfg.hidden, (cfg.Hq + 2 * cfg.Hkv) * cfg.D
    n = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    qkv = torch.empty((cfg.B, cfg.S, F), dtype=torch.bfloat16, device=dev)
    a = torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.S), dtype=torch.float32, device=dev)
    y = torch.empty_like(x)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    x2 = x.view(M, H)
    stages = [
        ("layernorm", lambda: A.layernorm(x2, gamma, beta, out=n, stream=stream)),
        ("qkv_gemm", lambda: A.linear(n, w_qkv, b_qkv, out=qkv.view(M, F), stream=stream)),
        ("attention", lambda: A.attention_qkvpacked(qkv, cfg.Hq, cfg.Hkv, cfg.D, causal=cfg.causal, out=a, lse=lse,
                                                    stream=stream)),
        ("out_gemm", lambda: A.linear(a.view(M, H), w_o, b_o, x2, out=y.view(M, H), stream=stream)),
    ]
    for _ in range(args.warmup):
        flush.zero_()
        for _, fn in stages:
            fn()
    torch.cuda.synchronize(dev)
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError("kernel reported a device timeout during warm-up")
    clocks = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError("kernel reported a device timeout in the timed region")
    per_stage = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)] for j in range(len(stages))]
    step_ms = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps)]
    max_s = reduce_max(sum(step_ms) / 1e3, dev)
    if rank == 0:
        clocks.stop()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    qkv_flops = 2.0 * M * F * H
    qkv_ms = statistics.median(per_stage[1])
    stage_flops = {"layernorm": 0.0, "qkv_gemm": qkv_flops, "out_gemm": 2.0 * M * H * H,
                   "attention": cfg.flops - qkv_flops - 2.0 * M * H * H}
    line = {
        "metric": "attention block fwd TFLOP/s (bf16): LayerNorm + QKV GEMM + causal attention + output GEMM + "
                  "residual", "value": whole_job_tflops(cfg.flops, args.steps, world, max_s), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "hidden": H, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                   "D": cfg.D, "causal": cfg.causal, "seed": cfg.seed,
                   "l2": "flushed before every timed step (untimed 256 MiB write)"},
        "roofline": {"bound": "tensor", "kernel": "gemm_bf16_kernel (QKV projection, M=%d N=%d K=%d)" % (M, F, H),
                     "achieved": qkv_flops / (qkv_ms / 1e3) / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": qkv_flops / (qkv_ms / 1e3) / 1e12 / peak,
                     "traffic": profiled_traffic("gemm_qkv_llama2_7b_block", "gemm"),
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "median_ms": qkv_ms},
        "stages": {name: {"median_ms": statistics.median(t),
                          "tflops": (stage_flops[name] / (statistics.median(t) / 1e3) / 1e12) if stage_flops[name]
                          else None} for (name, _), t in zip(stages, per_stage)},
        "gpu_launches": args.steps * len(stages),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "kernel_source_hash": kernel_source_hash("gemm"),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args):
    """Decode over a KV cache through the split-key entry point (attention + merge)."""
    from transformer_attention_02_gb300 import attn as A
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    A.lib()
    cfg = I.DECODE_CONFIGS[args.decode_config]
    q, k, v, _ = I.make_inputs(cfg)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.Sq), dtype=torch.float32, device=dev)
    splits = A.attn_splitkv_num_splits(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, 0)
    ws = torch.empty(max(1, A.attn_splitkv_workspace_bytes(cfg.B, cfg.Hq, cfg.Hkv, cfg.Sq, cfg.Sk, cfg.D, 0)),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def launch():
        A.attention_splitkv(qd, kd, vd, causal=cfg.causal, num_splits=0, workspace=ws, out=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        launch()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    if A.attn_last_status(stream.cuda_stream) != A.ATTN_OK:
        raise RuntimeError("kernel reported a device timeout in the timed region")
    ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    max_s = reduce_max(sum(ms) / 1e3, dev)
    if rank == 0:
        clocks.stop()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return 0
    nbytes = 2 * (q.numel() + k.numel() + v.numel() + o.numel()) + 4 * lse.numel()
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = nbytes * args.steps * world / max_s / 1e9
    med = statistics.median(ms)
    line = {
        "metric": "decode attention over a KV cache, GB/s of algorithmic bytes (split-key path)", "value": gbs,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {**config_json(cfg), "num_splits": splits},
        "roofline": {"bound": "hbm", "achieved": nbytes / (med / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": nbytes / (med / 1e3) / 1e9 / hbm, "traffic": None,
                     "peak_source": f"{peak_src} hbm_gbs", "kernel": "attn_fwd_kernel + splitkv_combine_kernel",
                     "median_ms": med},
        "gpu_launches": args.steps * (2 if splits > 1 else 1),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=I.BENCH_CONFIG, choices=sorted(I.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-configs", default="gqa_prefill,long_gqa_prefill",
                    help="more workloads timed after the headline one, reported under 'configs' "
                         "(comma-separated; empty for none)")
    ap.add_argument("--decode", action="store_true", help="decode over a KV cache (split-key path)")
    ap.add_argument("--decode-config", default="gqa_decode", choices=sorted(I.DECODE_CONFIGS))
    ap.add_argument("--block", action="store_true",
                    help="the attention block of one Llama-2-7B-sized layer (LayerNorm, projections, attention)")
    ap.add_argument("--rope", action="store_true",
                    help="rotary position embedding: keys rotated once per step, queries inside the kernel")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = I.CONFIGS[args.config]
    if args.block and args.impl != "reference":
        return run_block(args)
    if args.decode and args.impl != "reference":
        return run_decode(args)
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
