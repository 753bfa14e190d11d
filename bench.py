#!/usr/bin/env python
"""Benchmark of the paged GQA/MQA attention step on GB300.

One step = the whole hot path over one batch: reshape_and_cache of the
step's new K/V rows into the paged cache, then paged attention (decode, or
the mixed chunked-prefill + decode batch), all through the C ABI.

Headline workload (one GPU): Llama-3.1-8B-shaped decode -- 256 sequences,
32 query / 8 KV heads, head_dim 128, bf16, block 16, lognormal context
lengths (median 400, clipped to [16, 4096]).  Metric: KV-cache GB/s, the
algorithmic bytes sum_b ctx_b * Hkv * D * 2 (K and V) * 2 bytes over the
step time.  The mixed batch (64 sequences: 16 query chunks + 48 decode rows)
is reported beside it in tokens/s.

Inputs are synthetic and seeded (workloads/); under torchrun every rank runs
its own replica (the path has no exchange step), so scaling is weak.

--impl reference times the fp64 CPU oracle, as it stands, on the host cores
(a bounded sample of the same workload per step); it is the slow reference
arm of this benchmark, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged GQA decode KV-cache GB/s (% of GB300 HBM peak); mixed-batch tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode",
                    choices=["llama8b_decode", "mixed_prefill_decode", "head_sweep_kv1",
                             "head_sweep_kv8", "head_sweep_kv32", "long_context_decode",
                             "tiny_gqa_decode", "cross_attention_decode",
                             "cross_attention_prefill", "varlen_prefill_llama8b"],
                    help="varlen_prefill_llama8b times gqa_varlen_prefill alone (one GPU; "
                         "its prefill kernel's tensor roofline), for profiling that kernel")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the mixed-batch line item")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--block-size", type=int, default=16,
                    help="cache block size for llama8b_decode / mixed_prefill_decode "
                         "(the block-size sweep); 16 is the headline configuration")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--host-link", action="store_true",
                    help="only measure the host<->device copy rate of pinned buffers over a "
                         "range of sizes (the link the end-to-end figure's copies cross)")
    return ap.parse_args()


def make_workload(name: str, seed: int, block_size: int = 16):
    if name.startswith("head_sweep_kv"):
        return W.head_sweep(seed, num_kv_heads=int(name[len("head_sweep_kv"):]))
    if block_size != 16:
        if name not in ("llama8b_decode", "mixed_prefill_decode", "cross_attention_decode",
                        "cross_attention_prefill"):
            raise SystemExit("--block-size applies to llama8b_decode, mixed_prefill_decode "
                             "and the cross_attention workloads")
        return W.WORKLOADS[name](seed, block_size=block_size)
    return W.WORKLOADS[name](seed)


# ---------------------------------------------------------------- env helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def whole_job(units: float, step_s: float, e2e_s: float, world: int, device):
    """Whole-job figures of a replicated run (one process per GPU, each with
    its own seeded batch): the work units of all ranks summed, and each time
    the slowest rank's.  Collective over the default process group (NCCL on
    GPUs; any backend works, gloo on CPU in the tests)."""
    if world <= 1:
        return units, step_s, e2e_s
    import torch
    import torch.distributed as dist
    u = torch.tensor([units], device=device, dtype=torch.float64)
    t = torch.tensor([step_s, e2e_s], device=device, dtype=torch.float64)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u[0]), float(t[0]), float(t[1])


def measured_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s) measured for a kernel timed on its own."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s"


def prefill_flops(case) -> float:
    """QK^T and PV of the query chunks (qlen > 1): 4 * Hq * D per visible key
    (causal: token i of a chunk sees ctx - qlen + i + 1 keys; cross-attention:
    every row sees all ctx keys)."""
    ql = np.asarray(case.query_lens, dtype=np.int64)
    cl = np.asarray(case.context_lens, dtype=np.int64)
    cross = getattr(case, "cross", False)
    total = 0.0
    for q, c in zip(ql, cl):
        if q > 1:
            keys = q * c if cross else q * (c - q) + q * (q + 1) // 2
            total += 4.0 * case.num_heads * case.head_dim * float(keys)
    return total


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clk", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        smax = max(num(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": float(np.nanmedian(sm)), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows)}


def kernel_source_sha(fname: str) -> str:
    """Hash of a kernel's source file and the headers every kernel includes."""
    h = hashlib.sha256()
    for part in (fname, "pa_common.cuh", "pa_kernels.cuh"):
        with open(os.path.join(ROOT, "mqa_paged_kv_gb300", "csrc", part), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str, src_file: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/), or None
    when no capture matches the current kernel source and workload."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(src_file)
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if (parts.get("kernel") == kernel_key and parts.get("source_sha") == sha
                    and parts.get("workload") == workload):
                try:
                    return float(parts["bytes_per_launch"])
                except (KeyError, ValueError):
                    return None
    return None


def step_time_stats(ms) -> dict:
    """Summary of per-step times (ms), with every step's time so that an
    outlier step can be traced to its position in the run."""
    ms = np.asarray(ms, dtype=np.float64)
    return {"min_ms": float(ms.min()), "median_ms": float(np.median(ms)),
            "p90_ms": float(np.percentile(ms, 90)), "max_ms": float(ms.max()),
            "mean_ms": float(ms.mean()), "per_step_ms": [round(float(x), 5) for x in ms]}


def bench_config(case, args, world: int, *, host: bool, step_stats=None) -> dict:
    """The `config` of both arms, from one place and with the same keys: the
    workload's shape, the split policy, what one step is, and the timing
    fields (marked for the host-timed oracle arm)."""
    splits = getattr(args, "splits", 0)
    return dict(
        W.describe(case), splits=splits or "auto",
        step=("cross-attention over the static encoder cache" if case.cross
              else "reshape_and_cache + paged attention"),
        parallelism="single GPU" if world <= 1 else f"replicas x{world}",
        l2=("n/a (host)" if host else
            f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB read sweep)"),
        timing=("host perf_counter around each oracle step" if host else
                "CUDA events around each step on the launching stream; the host enqueues all "
                "timed steps while a blocking kernel holds the GPU, so no host launch gap "
                "falls inside a step"),
        step_time_stats=step_stats)


# ---------------------------------------------------------------- CPU arms
def oracle_sample_rows(case, target_s: float, threads: int):
    """Pick a prefix of query rows whose oracle run takes about target_s."""
    import oracle
    T = case.total_query_tokens
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping)
    rng = np.random.default_rng(1234)
    order = rng.permutation(T)
    n = max(1, min(T, 8))
    while True:
        rows = np.sort(order[:n])
        t0 = time.perf_counter()
        oracle.paged_attention(case.q, kc, vc, case.block_tables, case.cu_query_lens,
                               case.context_lens, case.scale, case.num_kv_heads, case.dtype,
                               rows=rows, num_threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or n >= T:
            break
        n = min(T, int(n * max(2.0, target_s / max(dt, 1e-3))))
    return rows, kc, vc


def sample_kv_bytes(case, rows):
    """KV bytes the attention of `rows` reads (each row's visible keys, once
    per KV head), the same algorithmic count as the GPU metric."""
    cu = case.cu_query_lens
    b_of = np.searchsorted(cu, rows, side="right") - 1
    ctx = case.context_lens[b_of].astype(np.int64)
    ql = (cu[b_of + 1] - cu[b_of]).astype(np.int64)
    pos = ctx - ql + (rows - cu[b_of])
    if case.is_decode:
        keys = ctx
    else:
        keys = pos + 1
    return int(keys.sum()) * case.num_kv_heads * case.head_dim * 2 * case.elem_bytes


def run_oracle_timed(case, rows, kc, vc, threads, reps=1):
    import oracle
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_attention(case.q, kc, vc, case.block_tables, case.cu_query_lens,
                               case.context_lens, case.scale, case.num_kv_heads, case.dtype,
                               rows=rows, num_threads=threads)
    return (time.perf_counter() - t0) / reps


def cpu_baseline(case, target_s=12.0):
    import oracle
    threads = os.cpu_count() or 1
    rows, kc, vc = oracle_sample_rows(case, target_s / 3, threads)
    dt = run_oracle_timed(case, rows, kc, vc, threads)
    kvb = sample_kv_bytes(case, rows)
    return {"value": kvb / dt / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{len(rows)} of {case.total_query_tokens} query rows of {case.name} "
                      f"(all heads), {dt:.2f} s, fp64 OpenMP C"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    case = make_workload(args.workload, args.seed, args.block_size)
    threads = os.cpu_count() or 1
    rows, kc, vc = oracle_sample_rows(case, 2.0, threads)
    kvb = sample_kv_bytes(case, rows)
    for _ in range(args.warmup):
        run_oracle_timed(case, rows, kc, vc, threads)
    times = np.array([run_oracle_timed(case, rows, kc, vc, threads)
                      for _ in range(max(1, args.steps))])
    dt = float(times.mean())
    step_stats = step_time_stats(times * 1e3)
    value = kvb / dt / 1e9
    sample = (f"{len(rows)} of {case.total_query_tokens} query rows of {case.name} per step "
              f"(all heads), fp64 OpenMP C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(case, args, world, host=True, step_stats=step_stats),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
class Step:
    """Device-resident inputs of one workload and its step through the C ABI."""

    def __init__(self, case, device, splits):
        import torch
        import mqa_paged_kv_gb300 as pa
        self.torch, self.pa, self.case, self.splits = torch, pa, case, splits
        et = torch.float16 if case.dtype == W.F16 else torch.bfloat16
        self.et = et

        def dev(a, dt=None):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                t = t.view(torch.int16).view(dt)
            return t.to(device)

        self.dev = dev
        self.k_cache = dev(case.k_cache, et)
        self.v_cache = dev(case.v_cache, et)
        self.inputs = {
            "q": dev(case.q, et), "k_new": dev(case.k_new, et), "v_new": dev(case.v_new, et),
            "slot_mapping": dev(case.slot_mapping), "block_tables": dev(case.block_tables),
            "context_lens": dev(case.context_lens), "cu_query_lens": dev(case.cu_query_lens),
        }
        self.out = torch.empty_like(self.inputs["q"])
        if case.is_decode and not case.cross:
            nb = pa.paged_attn_workspace_bytes(case.num_seqs, case.num_heads,
                                               case.num_kv_heads, case.head_dim,
                                               case.max_blocks_per_seq, case.block_size, splits)
        else:
            nb = pa.paged_attn_chunked_prefill_workspace_bytes(
                case.num_seqs, case.total_query_tokens, case.num_heads, case.num_kv_heads,
                case.head_dim, case.max_blocks_per_seq, case.block_size, splits)
        self.ws = pa.alloc_workspace(nb, device)
        self.launches = 0

    def run(self, x=None, prof=None):
        pa, c = self.pa, self.case
        x = x or self.inputs
        n = 0
        if not c.cross:  # a cross-attention encoder cache is static: nothing to write
            pa.reshape_and_cache(x["k_new"], x["v_new"], self.k_cache, self.v_cache,
                                 x["slot_mapping"])
            n = pa.last_launch_count()
        if prof is not None:
            pa.pa_profile_next_call(*prof)
        if c.cross:
            pa.paged_attn_cross_attention(x["q"], self.k_cache, self.v_cache,
                                          x["block_tables"], x["cu_query_lens"],
                                          x["context_lens"], c.max_query_len, c.scale,
                                          out=self.out, num_splits=self.splits,
                                          workspace=self.ws)
        elif c.is_decode:
            pa.paged_attn_decode(x["q"], self.k_cache, self.v_cache, x["block_tables"],
                                 x["context_lens"], c.scale, out=self.out,
                                 num_splits=self.splits, workspace=self.ws)
        else:
            pa.paged_attn_chunked_prefill(x["q"], self.k_cache, self.v_cache, x["block_tables"],
                                          x["cu_query_lens"], x["context_lens"],
                                          c.max_query_len, c.scale, out=self.out,
                                          num_splits=self.splits, workspace=self.ws)
        n += pa.last_launch_count()
        self.launches += n
        return self.out


def hold_gpu(torch, seconds: float) -> None:
    """Enqueue a kernel that keeps the GPU busy for about `seconds`, so that
    the host can enqueue the timed steps behind it and the device never
    waits for the host inside a step (the blocking-kernel method of
    GPU benchmark harnesses).  The kernel spins on the SM clock for a fixed
    count, so it always ends."""
    torch.cuda._sleep(int(max(seconds, 1e-4) * 2.5e9))


def time_steps(step, steps, warmup, flush, e2e=False):
    """Per-step CUDA-event times (ms) of the step and of its attention kernels;
    L2 is flushed before every timed step, outside the timed interval.  The
    host enqueues all timed steps while a blocking kernel holds the GPU."""
    torch = step.torch
    stream = torch.cuda.current_stream()
    host_pack = dev_pack = dev_bufs = None
    if e2e:
        # The step's inputs travel as one pinned host buffer and one copy
        # (tensors at 256-byte aligned offsets, device views into one buffer).
        offs, off = {}, 0
        for k, v in step.inputs.items():
            offs[k] = off
            off += (v.numel() * v.element_size() + 255) // 256 * 256
        host_pack = torch.empty(max(off, 256), dtype=torch.uint8).pin_memory()
        dev_pack = torch.empty(max(off, 256), dtype=torch.uint8, device=step.out.device)
        dev_bufs = {}
        for k, v in step.inputs.items():
            nb = v.numel() * v.element_size()
            if nb == 0:  # an empty input (no new K/V in a cross-attention step)
                dev_bufs[k] = torch.empty_like(v)
                continue
            host_pack[offs[k]:offs[k] + nb].copy_(
                v.contiguous().reshape(-1).view(torch.uint8).cpu())
            dev_bufs[k] = dev_pack[offs[k]:offs[k] + nb].view(v.dtype).view(v.shape)
        out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()

    def one(prof=None):
        if e2e:
            dev_pack.copy_(host_pack, non_blocking=True)
            o = step.run(dev_bufs, prof)
            out_host.copy_(o, non_blocking=True)
        else:
            step.run(None, prof)

    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(warmup):
        flush.sum()
        one()
    host_per_step = (time.perf_counter() - h0) / max(1, warmup)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    hold_s = min(0.5, 2.0 * steps * host_per_step + 2e-3)
    step.launches = 0
    hold_gpu(torch, hold_s)
    for i in range(steps):
        flush.sum()  # read-only sweep: evicts L2 without leaving dirty lines behind
        e0, e1, _, _ = ev[i]
        e0.record(stream)
        one()
        e1.record(stream)
    torch.cuda.synchronize()
    launches = step.launches
    # second pass: the attention kernels alone, bracketed by events the
    # library records around them (kept out of the step timing above, where
    # extra events would sit between the chained launches)
    hold_gpu(torch, hold_s)
    for i in range(steps):
        flush.sum()
        _, _, k0, k1 = ev[i]
        one((k0, k1))
    torch.cuda.synchronize()
    step.launches = launches
    t = np.array([a.elapsed_time(b) for a, b, _, _ in ev])
    kt = np.array([c.elapsed_time(d) for _, _, c, d in ev])
    h2d = sum(v.numel() * v.element_size() for v in step.inputs.values()) if e2e else 0
    d2h = step.out.numel() * step.out.element_size() if e2e else 0
    if e2e:
        # the two copies alone (same buffers, same stream), so the step's
        # end-to-end cost can be split into link time and the rest
        cev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        hold_gpu(torch, min(0.5, steps * 2e-4 + 2e-3))
        for e in cev:
            e[0].record(stream)
            dev_pack.copy_(host_pack, non_blocking=True)
            e[1].record(stream)
            e[2].record(stream)
            out_host.copy_(step.out, non_blocking=True)
            e[3].record(stream)
        torch.cuda.synchronize()
        h2d_ms = float(np.median([e[0].elapsed_time(e[1]) for e in cev]))
        d2h_ms = float(np.median([e[2].elapsed_time(e[3]) for e in cev]))
        time_steps.copy_only = {
            "h2d_ms": h2d_ms, "d2h_ms": d2h_ms,
            "h2d_gbs": dev_pack.numel() / (h2d_ms / 1e3) / 1e9,
            "d2h_gbs": d2h / (d2h_ms / 1e3) / 1e9,
            "note": "median over steps of each copy alone (pinned host memory, one "
                    "cudaMemcpyAsync each), CUDA events on the step's stream"}
    return t, kt, h2d, d2h


def decode_roofline(case, kern_s: float) -> dict:
    """HBM roofline of decode_kernel: the algorithmic KV bytes (each context
    token's K and V rows once per KV head) over the kernel's live duration."""
    kvb = case.kv_bytes()
    peak, peak_src = measured_hbm_peak()
    achieved = kvb / kern_s / 1e9
    traffic = ncu_traffic("decode_kernel", "decode.cu", case.name)
    return {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved,
            "peak": peak, "peak_source": peak_src, "unit": "GB/s",
            "frac": achieved / peak, "kernel_ms": kern_s * 1e3,
            "algorithmic_bytes": kvb, "traffic": traffic,
            "traffic_ratio": (traffic / kvb) if traffic else None}


def measure_decode(case, device, splits: int, steps: int, warmup: int, flush,
                   cpu: bool = False) -> dict:
    """One decode configuration: step time (cache write + attention call),
    the decode kernel's live time and its HBM roofline; with cpu, also the
    oracle on a bounded sample of the same workload (host cores)."""
    st = Step(case, device, splits)
    t, kt, _, _ = time_steps(st, steps, warmup, flush)
    del st
    ms = float(t.mean())
    extra = {}
    if cpu:
        try:
            extra["cpu_baseline"] = cpu_baseline(case, target_s=3.0)
        except Exception as e:  # reported, never required
            extra["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
    return {**extra, "kv_bytes": case.kv_bytes(), "ms_per_step": ms,
            "step_gbs": case.kv_bytes() / (ms / 1e3) / 1e9,
            "tokens_per_s": case.total_query_tokens / (ms / 1e3),
            "step_time_stats": step_time_stats(t),
            "roofline": decode_roofline(case, float(kt.mean()) / 1e3),
            "splits": splits or "auto"}


def measure_other_decode_configs(seed: int, device, steps: int, warmup: int, flush,
                                 cpu: bool = False) -> dict:
    """The other decode configurations of the benchmark, each with its own
    roofline: the tiny GQA decode (a latency figure), the MQA / GQA / MHA
    sweep at 32 query heads (side by side: KV bytes, tokens/s, kernel
    fraction of HBM peak, recorded DRAM traffic), and long-context split-KV
    decode with automatic and fixed split counts."""
    res = {}
    tiny = W.tiny_gqa_decode(seed)
    r = measure_decode(tiny, device, 0, steps, warmup, flush, cpu)
    r["latency_us"] = r["ms_per_step"] * 1e3
    r["note"] = ("latency-bound: 0.3 MB of KV; the roofline fraction is reported for "
                 "completeness, the step latency is the figure")
    res["tiny_gqa_decode"] = r
    sweep = {}
    for hkv in (1, 8, 32):
        c = W.head_sweep(seed, num_kv_heads=hkv)
        sweep[f"kv{hkv}"] = dict(measure_decode(c, device, 0, steps, warmup, flush, cpu),
                                 num_kv_heads=hkv, G=c.num_heads // hkv)
        del c
    res["head_sweep"] = sweep
    lc = W.long_context_decode(seed)
    res["long_context_decode"] = {
        ("auto" if s == 0 else str(s)): measure_decode(lc, device, s, steps, warmup, flush,
                                                       cpu and s == 0)
        for s in (0, 16, 32, 64)}
    return res


def prefill_roofline(workload: str, seed: int, device, args, flush):
    """Tensor roofline of prefill_tc_kernel on the query chunks of a mixed
    batch: the chunks alone (same lengths, seed and shapes, no decode rows)
    are timed through the same call, so the kernel hook brackets only the
    prefill kernel (and an empty decode launch)."""
    pcase = W.mixed_prefill_decode(seed, n_decode=0, block_size=args.block_size)
    pstep = Step(pcase, device, args.splits)
    _, pkt, _, _ = time_steps(pstep, max(5, args.steps // 2), 3, flush)
    del pstep
    flops = prefill_flops(pcase)
    kern_s = float(pkt.mean()) / 1e3
    peak, src = measured_bf16_peak()
    achieved = flops / kern_s / 1e12
    return {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": achieved,
            "peak": peak, "peak_source": src, "unit": "TFLOP/s", "frac": achieved / peak,
            "kernel_ms": kern_s * 1e3, "algorithmic_flops": flops,
            "traffic": ncu_traffic("prefill_tc_kernel", "prefill_tc.cu", workload),
            "timed_on": f"the {pcase.num_seqs} query chunks of {workload} (seed {seed}) alone"}


def graph_replay_times(step, steps: int, warmup: int, flush):
    """The step (cache write + attention call) captured once in a CUDA graph
    on a side stream and replayed: CUDA-event time of each replay (ms), L2
    swept before each, outside the timed interval."""
    torch = step.torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # the first calls set kernel attributes: not in a capture
        step.run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step.run()
    torch.cuda.synchronize()
    for _ in range(warmup):
        flush.sum()
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    hold_gpu(torch, min(0.5, steps * 3e-4 + 2e-3))
    for a, b in ev:
        flush.sum()
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    del graph
    return np.array([a.elapsed_time(b) for a, b in ev])


def measure_graph_steps(seed: int, device, steps: int, warmup: int, flush) -> dict:
    """Decode steps replayed from a CUDA graph (the way a serving loop issues
    a fixed-shape step): the headline batch and the latency-bound tiny one."""
    res = {}
    for name in ("llama8b_decode", "tiny_gqa_decode"):
        case = make_workload(name, seed)
        step = Step(case, device, 0)
        t = graph_replay_times(step, steps, warmup, flush)
        del step
        ms = float(t.mean())
        res[name] = {"ms_per_step": ms, "median_ms": float(np.median(t)),
                     "step_gbs": case.kv_bytes() / (ms / 1e3) / 1e9,
                     "tokens_per_s": case.total_query_tokens / (ms / 1e3)}
    res["note"] = ("cache write + decode call captured once in a CUDA graph and replayed; "
                   "CUDA events around each replay, L2 swept before each")
    return res


def measure_varlen(seed: int, device, steps: int, warmup: int, flush):
    """gqa_varlen_prefill on the Llama-3.1-8B prompt batch (16 prompts of
    U[128, 2048] tokens, contiguous K/V, no cache): CUDA-event time of the
    whole call and of its prefill kernel, tensor roofline of the kernel."""
    import torch
    import mqa_paged_kv_gb300 as pa
    c = W.varlen_prefill_llama8b(seed)
    et = torch.bfloat16

    def dev(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(dt)
        return t.to(device)
    q, k, v = dev(c.q, et), dev(c.k, et), dev(c.v, et)
    cq, ck = dev(c.cu_q), dev(c.cu_k)
    out = torch.empty_like(q)
    ws = pa.alloc_workspace(pa.gqa_varlen_prefill_workspace_bytes(
        c.num_seqs, c.total_query_tokens, c.num_heads, c.num_kv_heads, c.head_dim), device)

    def call(prof=None):
        if prof is not None:
            pa.pa_profile_next_call(*prof)
        pa.gqa_varlen_prefill(q, k, v, cq, ck, c.max_query_len, c.scale, out=out, workspace=ws)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    hold_gpu(torch, min(0.5, steps * 4e-4 + 2e-3))
    for e in ev:
        flush.sum()
        e[0].record(stream)
        call()
        e[1].record(stream)
    hold_gpu(torch, min(0.5, steps * 4e-4 + 2e-3))
    for e in ev:
        flush.sum()
        call((e[2], e[3]))
    torch.cuda.synchronize()
    t = float(np.mean([e[0].elapsed_time(e[1]) for e in ev])) / 1e3
    kt = float(np.mean([e[2].elapsed_time(e[3]) for e in ev])) / 1e3
    flops = c.flops()
    peak, src = measured_bf16_peak()
    ach = flops / kt / 1e12
    return {"tokens_per_s": c.total_query_tokens / t, "ms_per_step": t * 1e3,
            "query_tokens": c.total_query_tokens,
            "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": ach,
                         "peak": peak, "peak_source": src, "unit": "TFLOP/s",
                         "frac": ach / peak, "kernel_ms": kt * 1e3, "algorithmic_flops": flops,
                         "traffic": ncu_traffic("prefill_tc_kernel", "prefill_tc.cu",
                                                "varlen_prefill_llama8b")}}


def run_varlen_only(args):
    """The varlen prompt batch alone on one GPU: its call and prefill-kernel
    times and the kernel's tensor roofline, as one JSON line."""
    import torch
    _, world, _ = dist_env()
    if world > 1 or args.impl == "reference":
        raise SystemExit("varlen_prefill_llama8b runs on one GPU with --impl ours only")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    import mqa_paged_kv_gb300  # noqa: F401  (fails loudly when the library is missing)
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    res = measure_varlen(args.seed, device, args.steps, max(3, args.warmup), flush)
    clocks = clk.stop()
    r = res["roofline"]
    print(json.dumps({
        "metric": "varlen prompt prefill attention TFLOP/s", "value": r["achieved"],
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "varlen_prefill_llama8b", "query_tokens": res["query_tokens"],
                   "l2": "flushed before every timed call (256 MiB read sweep)"},
        "tokens_per_s": res["tokens_per_s"], "roofline": r, "clocks": clocks}), flush=True)


def measure_two_kernel(seed: int, device, steps: int, warmup: int, flush, block_size: int = 16):
    """The mixed batch two ways, attention only, cache already written:
    (a) the library's one call (one work list; the prefill kernel and the
    decode kernel resident side by side, the decode kernel on the SM share
    the work list gives it and on each SM the prefill kernel frees); (b) the
    arrangement of vLLM PR #14431's op: a
    prefill call over the query chunks only and a decode call over the
    decode rows on a second stream, concurrently, with the SMs split between
    them (pa_limit_next_call_ctas); every split in `splits` is timed."""
    import torch
    import mqa_paged_kv_gb300 as pa
    c = W.mixed_prefill_decode(seed, block_size=block_size)
    et = torch.bfloat16

    def dev(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(dt)
        return t.to(device)
    kc, vc = dev(c.k_cache, et), dev(c.v_cache, et)
    pa.reshape_and_cache(dev(c.k_new, et), dev(c.v_new, et), kc, vc, dev(c.slot_mapping))
    q_all = dev(c.q, et)
    cu = np.asarray(c.cu_query_lens)
    ql = np.diff(cu)
    pre, dec = np.where(ql > 1)[0], np.where(ql == 1)[0]
    rows_p = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in pre])
    q_p, q_d = dev(c.q[rows_p], et), dev(c.q[cu[dec]], et)
    cu_p = np.zeros(len(pre) + 1, np.int32)
    cu_p[1:] = np.cumsum(ql[pre])
    bt, ctx = np.asarray(c.block_tables), np.asarray(c.context_lens)
    t_all = {"bt": dev(bt), "ctx": dev(ctx), "cu": dev(cu.astype(np.int32))}
    t_p = {"bt": dev(bt[pre]), "ctx": dev(ctx[pre]), "cu": dev(cu_p)}
    t_d = {"bt": dev(bt[dec]), "ctx": dev(ctx[dec])}
    o_all, o_p, o_d = torch.empty_like(q_all), torch.empty_like(q_p), torch.empty_like(q_d)
    H, Hkv, D, mbs = c.num_heads, c.num_kv_heads, c.head_dim, c.max_blocks_per_seq
    ws_all = pa.alloc_workspace(pa.paged_attn_chunked_prefill_workspace_bytes(
        c.num_seqs, c.total_query_tokens, H, Hkv, D, mbs, c.block_size, 0), device)
    ws_p = pa.alloc_workspace(pa.paged_attn_chunked_prefill_workspace_bytes(
        len(pre), len(rows_p), H, Hkv, D, mbs, c.block_size, 0), device)
    ws_d = pa.alloc_workspace(pa.paged_attn_workspace_bytes(
        len(dec), H, Hkv, D, mbs, c.block_size, 0), device)
    main = torch.cuda.current_stream()
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count

    def fused():
        pa.paged_attn_chunked_prefill(q_all, kc, vc, t_all["bt"], t_all["cu"], t_all["ctx"],
                                      c.max_query_len, c.scale, out=o_all, workspace=ws_all)

    def two(k):
        fork = torch.cuda.Event()
        fork.record(main)
        s1.wait_event(fork)
        s2.wait_event(fork)
        pa.pa_limit_next_call_ctas(sms - k if k else 0)
        pa.paged_attn_chunked_prefill(q_p, kc, vc, t_p["bt"], t_p["cu"], t_p["ctx"],
                                      c.max_query_len, c.scale, out=o_p, workspace=ws_p,
                                      stream=s1)
        pa.pa_limit_next_call_ctas(k)
        pa.paged_attn_decode(q_d, kc, vc, t_d["bt"], t_d["ctx"], c.scale, out=o_d,
                             workspace=ws_d, stream=s2)
        j1, j2 = torch.cuda.Event(), torch.cuda.Event()
        j1.record(s1)
        j2.record(s2)
        main.wait_event(j1)
        main.wait_event(j2)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = []
        hold_gpu(torch, min(0.5, steps * 6e-4 + 2e-3))
        for _ in range(steps):
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            fn()
            b.record(main)
            ev.append((a, b))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ev]))
    res = {"fused_ms": timed(fused), "two_kernel_ms": {}}
    for k in (0, 24, 40, 56, 72):
        res["two_kernel_ms"][str(k) if k else "no split"] = timed(lambda: two(k))
    best = min(res["two_kernel_ms"], key=res["two_kernel_ms"].get)
    res["best_two_kernel"] = {"decode_sms": best, "ms": res["two_kernel_ms"][best]}
    res["note"] = ("attention only (cache written beforehand), median over steps; decode_sms = "
                   "SMs given to the decode call, the prefill call gets the rest")
    return res


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import mqa_paged_kv_gb300  # noqa: F401  (fails loudly when the library is missing)

    case = make_workload(args.workload, args.seed + rank, args.block_size)
    step = Step(case, device, args.splits)
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    clk = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk.start()
    wall0 = time.perf_counter()
    t, kt, _, _ = time_steps(step, args.steps, args.warmup, flush)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = clk.stop()
    launches = step.launches

    te, _, h2d, d2h = time_steps(step, max(3, args.steps // 2), max(3, args.warmup), flush,
                                 e2e=True)
    del step

    kern_s = float(kt.mean()) / 1e3
    kvb = case.kv_bytes()
    job_kvb, step_s, e2e_s = whole_job(float(kvb), float(t.mean()) / 1e3, float(te.mean()) / 1e3,
                                       world, device)
    job_tokens, _, _ = whole_job(float(case.total_query_tokens), 0.0, 0.0, world, device)
    units = "GB/s"
    value = job_kvb / step_s / 1e9
    peak, _ = measured_hbm_peak()
    if case.is_decode:  # also cross-attention decode: the same decode kernel
        roofline = decode_roofline(case, kern_s)
    elif case.cross:  # every sequence carries a chunk: the call is the prefill kernel
        flops = prefill_flops(case)
        bpeak, bsrc = measured_bf16_peak()
        ach = flops / kern_s / 1e12
        roofline = {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": ach,
                    "peak": bpeak, "peak_source": bsrc, "unit": "TFLOP/s",
                    "frac": ach / bpeak, "kernel_ms": kern_s * 1e3,
                    "algorithmic_flops": flops,
                    "traffic": ncu_traffic("prefill_tc_kernel", "prefill_tc.cu", case.name)}
    else:
        roofline = prefill_roofline(args.workload, args.seed + rank, device, args, flush)

    line = {
        "metric": METRIC, "value": value, "unit": units, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if case.dtype == W.BF16 else "f16", "data": "synthetic",
        "config": bench_config(case, args, world, host=False, step_stats=step_time_stats(t)),
        "hbm_peak_frac": value / world / peak,
        "tokens_per_s": job_tokens / step_s,
        "roofline": roofline,
        "e2e": {"value": job_kvb / e2e_s / 1e9, "unit": units, "ms_per_step": e2e_s * 1e3,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "step_time_stats": step_time_stats(te),
                "copies_alone": getattr(time_steps, "copy_only", None)},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }

    sec_steps, sec_warm = max(10, args.steps), max(3, args.warmup)
    if not args.no_secondary and args.workload == "llama8b_decode":
        mcase = W.mixed_prefill_decode(args.seed + rank, block_size=args.block_size)
        mstep = Step(mcase, device, args.splits)
        mt, mkt, _, _ = time_steps(mstep, max(5, args.steps // 2), 3, flush)
        ms = float(mt.mean()) / 1e3
        del mstep
        line["secondary"] = {"mixed_prefill_decode": {
            "tokens_per_s": mcase.total_query_tokens / ms, "ms_per_step": ms * 1e3,
            "attention_kernels_ms": float(mkt.mean()),
            "kv_gbs": mcase.kv_bytes() / ms / 1e9, "query_tokens": mcase.total_query_tokens,
            "roofline": prefill_roofline("mixed_prefill_decode", args.seed + rank, device,
                                         args, flush)}}
        line["secondary"]["mixed_prefill_decode"]["two_kernel_comparison"] = measure_two_kernel(
            args.seed + rank, device, max(5, args.steps // 2), 3, flush, args.block_size)
        line["secondary"]["varlen_prefill_llama8b"] = measure_varlen(
            args.seed + rank, device, max(5, args.steps // 2), 3, flush)
        line["secondary"].update(measure_other_decode_configs(
            args.seed + rank, device, sec_steps, sec_warm, flush,
            cpu=rank == 0 and world == 1 and not args.no_cpu_baseline))
        line["secondary"]["graph_replay"] = measure_graph_steps(
            args.seed + rank, device, sec_steps, sec_warm, flush)

    if rank == 0 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline(case)
        except Exception as e:  # the baseline is reported, never required
            line["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def host_link_rates():
    """One cudaMemcpyAsync per direction between a pinned host buffer and
    device memory, over sizes around a decode step's inputs and outputs and
    up to where the rate saturates; median of 20 CUDA-event timings each."""
    import torch
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    rows = []
    for mb in (0.5, 2.1, 3.4, 16, 64, 256):
        n = int(mb * (1 << 20))
        h = torch.empty(n, dtype=torch.uint8).pin_memory()
        d = torch.empty(n, dtype=torch.uint8, device=dev)
        res = {"bytes": n}
        for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)),
                         ("d2h", lambda: h.copy_(d, non_blocking=True))):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            ev = []
            for _ in range(20):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev.append((a, b))
            torch.cuda.synchronize()
            ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
            res[name + "_us"] = ms * 1e3
            res[name + "_gbs"] = n / (ms / 1e3) / 1e9
        rows.append(res)
    print(json.dumps({"host_link": rows}), flush=True)


def main():
    args = parse_args()
    if args.host_link:
        host_link_rates()
        return
    if args.workload == "varlen_prefill_llama8b":
        run_varlen_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
