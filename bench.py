#!/usr/bin/env python
"""Benchmark of the GroupQueryAttention forward pass; prints one JSON line.

A step is one forward call (append + attention over the cache) on one batch
of synthetic input of the named workload, inputs resident in HBM. Default
workload: fp16 decode, B=16, N=32, N_kv=8, H=128, shared cache of capacity
8192, seqlens_k ~ U[1024, 8191], rotary (the configuration the metric is
quoted on). The metric for a decode workload is KV-cache bytes read per
second (GB/s, only the live rows); for a prefill workload it is attention
TFLOP/s (4*H per visible query/key pair).

--impl reference times the CPU oracle (fp64 numpy) on the host cores on a
bounded sample of the same workload.
The headline line (value, roofline, e2e, clocks, cpu_baseline) is the
default workload; the same measurements of the other configurations (tiny
fp32 prompt, fp16 causal prefill, fp16 chunked prefill, fp32 decode over an
int8 cache) follow under "workloads" (--workloads none skips them).
Under torchrun (N>1) every rank runs an independent replica on its own GPU
(the operator has no cross-GPU exchange); value = units of all ranks / max time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from grouped_query_attention_gb300.inputs import WORKLOADS, generate  # noqa: E402

METRIC = "decode KV-cache GB/s & prefill TFLOP/s, as fraction of GB300 roofline"
DEFAULT_WORKLOAD = "decode_f16_b16_c8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 CUDA-core peak: 152 SMs x 128 fp32 FMA lanes x 2 flop per clock at the maximum SM clock.
FP32_LANES_PER_SM, SM_COUNT = 128, 152
L2_FLUSH_BYTES = 512 << 20


# --------------------------------------------------------------------------- work accounting

def visible_pairs(case) -> tuple[int, int]:
    """(visible query/key pairs over all heads, live KV rows over all KV heads)."""
    inp, at = case["inputs"], case["attrs"]
    B, S = inp["query"].shape[:2]
    N, Nkv = at["num_heads"], at["kv_num_heads"]
    W = at["local_window_size"]
    has_past = inp.get("past_key") is not None
    pairs = 0
    kv_rows = 0
    for b in range(B):
        total = int(inp["seqlens_k"][b]) + 1
        past = total - S if has_past else 0
        live = S if has_past else min(S, total)
        p = past + np.arange(live)
        hi = np.minimum(p, total - 1) if at["causal"] else np.full(live, total - 1)
        lo = np.maximum(0, p - W) if W >= 0 else np.zeros(live, dtype=np.int64)
        pairs += int(np.sum(hi - lo + 1)) * N
        kstart = max(0, past - W) if W >= 0 else 0
        kv_rows += (total - kstart) * Nkv
    return pairs, kv_rows


def window_shift_bytes(case) -> int:
    """Bytes the window shift of a sliding-window cache reads and writes (K and V):
    the kept rows min(n_old + S, C) - S move unless they are already at the front."""
    sp, inp = case["spec"], case["inputs"]
    S, C = sp.S, sp.capacity
    L = C if sp.mode == "shared" else sp.past_len
    esize = 1 if sp.quant != "NONE" else (2 if sp.dtype == "f16" else 4)
    moved = 0
    for b in range(sp.B):
        past = int(inp["seqlens_k"][b]) + 1 - S
        n_old = min(past, L)
        keep = min(n_old + S, C) - S
        if sp.mode != "shared" or n_old - keep > 0:
            moved += keep
    return 2 * 2 * moved * sp.Nkv * sp.H * esize


def work(case) -> dict:
    sp = case["spec"]
    pairs, kv_rows = visible_pairs(case)
    esize = (0.5 if sp.bits == 4 else 1) if sp.quant != "NONE" else (2 if sp.dtype == "f16" else 4)
    kv_bytes = int(kv_rows * sp.H * 2 * esize)
    flops = 4.0 * sp.H * pairs
    decode = sp.S * (sp.N // sp.Nkv) <= 8
    if decode:
        return dict(kind="decode", unit="GB/s", units=kv_bytes / 1e9, kv_bytes=kv_bytes, flops=flops,
                    bound="hbm")
    return dict(kind="prefill", unit="TFLOP/s", units=flops / 1e12, kv_bytes=kv_bytes, flops=flops,
                bound="tensor")


# --------------------------------------------------------------------------- helpers

def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def source_sha(files) -> str:
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, "grouped_query_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel_src: list[str]):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("source_sha") != source_sha(kernel_src):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling while the GPU is busy."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("GQA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- oracle timing

def oracle_sample(case, budget_s: float, max_runs: int | None = None) -> dict:
    """Time the oracle on whole batch entries of the workload until `budget_s` elapses."""
    import oracle
    sp = case["spec"]
    inp = case["inputs"]
    wk = work(case)
    B = sp.B
    # One run = the oracle on batch entries 0..nb-1 (all heads, all rows) for decode;
    # for prefill, all rows of the first query heads of batch 0.
    if wk["kind"] == "decode":
        nb = B
        sub = _slice_batches(case, nb)
        sample_desc = f"all {nb} batch entries (every head and cache row), one full forward per run"
        run = lambda: oracle.gqa_forward(sub["inputs"], sub["attrs"], sub["present_key"], sub["present_value"],
                                         sub["share_buffer"])
        units = work(sub)["units"]
    else:
        heads = 2
        sub = _slice_batches(case, 1)
        S = sp.S
        samp = [(0, h, i) for h in range(heads) for i in range(S)]
        sample_desc = f"batch entry 0, query heads 0..{heads - 1}, all {S} rows (cache append in full)"
        run = lambda: oracle.gqa_forward(sub["inputs"], sub["attrs"], sub["present_key"], sub["present_value"],
                                         sub["share_buffer"], sample=samp)
        pairs_all, _ = visible_pairs(sub)
        units = 4.0 * sp.H * pairs_all / sp.N * heads / 1e12
    t0, c0 = time.perf_counter(), time.process_time()
    runs = 0
    while True:
        run()
        runs += 1
        if time.perf_counter() - t0 >= budget_s or (max_runs and runs >= max_runs):
            break
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return dict(value=units * runs / wall, unit=wk["unit"], cores=max(1, round(cpu / wall)), sample=sample_desc,
                seconds=wall, runs=runs, kind="oracle")


def _slice_batches(case, nb: int) -> dict:
    inp = case["inputs"]
    sub_inp = {}
    for k, v in inp.items():
        if v is None:
            continue
        if k in ("query", "key", "value", "past_key", "past_value", "seqlens_k"):
            sub_inp[k] = v[:nb]
        elif k == "attention_bias" and v.shape[0] > 1:
            sub_inp[k] = v[:nb]
        else:
            sub_inp[k] = v
    sub = dict(case)
    sub["inputs"] = sub_inp
    sub["present_key"] = None if case["present_key"] is None else case["present_key"][:nb]
    sub["present_value"] = None if case["present_value"] is None else case["present_value"][:nb]
    return sub


# --------------------------------------------------------------------------- GPU arm

def measure_workload(name: str, args, world: int, rank: int, local: int) -> dict:
    """Times one workload on this rank's GPU: device-resident steps (value, per-kernel events,
    roofline), the same steps end to end with host buffers (e2e), clocks, and on rank 0 at N=1
    the oracle on a bounded sample (cpu_baseline)."""
    import torch

    from grouped_query_attention_gb300 import GroupQueryAttention, capi

    device = torch.device("cuda", local)
    case = generate(WORKLOADS[name], seed=rank)
    sp = case["spec"]
    inp = case["inputs"]
    wk = work(case)

    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in inp.items()
           if v is not None and k != "total_sequence_length"}
    if case["share_buffer"]:
        pk, pv = dev["past_key"], dev["past_value"]
    else:
        pk = torch.from_numpy(case["present_key"]).to(device)
        pv = torch.from_numpy(case["present_value"]).to(device)
    opt = {k: dev[k] for k in ("past_key", "past_value", "cos_cache", "sin_cache", "attention_bias",
                               "head_sink", "k_scale", "v_scale", "q_norm_weight", "k_norm_weight") if k in dev}
    total_len = int(inp["total_sequence_length"][0])
    op = GroupQueryAttention(**case["attrs"])
    out = torch.empty_like(dev["query"])
    call = dict(query=dev["query"], key=dev["key"], value=dev["value"], seqlens_k=dev["seqlens_k"],
                total_sequence_length=total_len, present_key=pk, present_value=pv, output=out, **opt)
    plan = op.plan(**call)
    ws = torch.empty(max(int(plan.workspace_bytes), 256), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_words = flush.view(torch.float32)   # summed in place (no widening copy)

    def flush_l2():
        # Write a buffer larger than L2, then read it back, so that the timed
        # step starts with an L2 holding none of its data and no dirty lines.
        flush.zero_()
        flush_words.sum()
    stream = torch.cuda.current_stream(device)

    def step():
        op(workspace=ws, **call)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert op.device_status() == 0, f"{name}: device status set during warm-up"

    # Clock sampling: a short soak of the same step keeps the GPU busy while
    # nvidia-smi samples, then the K timed steps run inside the same window.
    sampler = ClockSampler(local)
    sampler.start()
    soak_end = time.perf_counter() + args.soak
    while time.perf_counter() < soak_end:
        for _ in range(20):
            flush_l2()
            step()
        torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush_l2()                         # L2 flush between timed iterations
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    # The same K steps again with per-kernel CUDA events (recorded by the
    # library around each launch on the launching stream): the roofline uses
    # the dominant kernel's time. Kept out of the pass above, whose step time
    # the event pairs between launches would lengthen.
    capi.gqa_profile_begin(op.handle, args.steps * int(plan.launches))
    for k in range(args.steps):
        flush_l2()
        step()
    torch.cuda.synchronize()
    launches = capi.gqa_profile_end(op.handle)
    barrier(world)
    clocks = sampler.stop()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    per_kernel = {}
    for kind, t in launches:
        per_kernel.setdefault(kind, []).append(t)
    dominant = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    dom_ms = max_over_ranks(sum(per_kernel[dominant]) / len(per_kernel[dominant]), world, device)
    ms_local = sum(times_ms) / len(times_ms)
    ms = max_over_ranks(ms_local, world, device)
    assert op.device_status() == 0, f"{name}: device status set during the timed steps"

    # ---- end to end through the public API with host buffers (pinned), copies in the timed region.
    # The step's inputs (query, key, value, seqlens_k) sit back to back in one pinned host buffer
    # and land with one copy in one device buffer whose views the call takes, as a serving loop
    # batches its small transfers; the output comes back with one copy.
    names = ("query", "key", "value", "seqlens_k")
    arrs = [np.ascontiguousarray(inp[k]) for k in names]
    offs, stage_bytes = [], 0
    for a in arrs:
        offs.append(stage_bytes)
        stage_bytes += (a.nbytes + 255) // 256 * 256
    host_stage = torch.empty(stage_bytes, dtype=torch.uint8).pin_memory()
    dev_stage = torch.empty(stage_bytes, dtype=torch.uint8, device=device)
    staged = {}
    for k, a, o in zip(names, arrs, offs):
        host_stage[o:o + a.nbytes].copy_(torch.from_numpy(a.reshape(-1).view(np.uint8)))
        staged[k] = dev_stage[o:o + a.nbytes].view(dev[k].dtype).view(dev[k].shape)
    call_e2e = dict(call, query=staged["query"], key=staged["key"], value=staged["value"],
                    seqlens_k=staged["seqlens_k"])
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = stage_bytes
    d2h = host_out.numel() * host_out.element_size()
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush_l2()
        e_starts[k].record(stream)
        dev_stage.copy_(host_stage, non_blocking=True)
        op(workspace=ws, **call_e2e)
        host_out.copy_(out, non_blocking=True)
        e_ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_starts, e_ends)) / args.steps, world, device)

    units_all = wk["units"] * world
    value = units_all / (ms / 1e3)
    e2e_value = units_all / (e2e_ms / 1e3)

    peaks, peaks_src = load_peaks()
    # The sources a kernel's code comes from (a traffic record holds only while they are unchanged).
    shared = ["common.cuh", "gqa_internal.h"]
    tc_decode_src = ["decode_tc.cu", "tcgen05.cuh"]
    tc_prefill_src = "prefill_tcq.cu" if sp.quant != "NONE" and sp.dtype == "f32" else "prefill_tc.cu"
    kernel_src = {"decode": ["decode.cu"], "decode_tensor_core": tc_decode_src,
                  "prefill_tensor_core": [tc_prefill_src, "tcgen05.cuh"],
                  "prefill_cuda_core": ["prefill_simt.cu"], "prepass": ["prepass.cu"],
                  "copy_past": ["prepass.cu"], "window_shift": ["prepass.cu"],
                  "bias_stage": ["prepass.cu"]}[dominant] + shared
    peak_key = "hbm_gbs" if wk["bound"] == "hbm" else "bf16_tflops"
    latency_bound = wk["units"] * 1e12 < 1e9 if wk["kind"] == "prefill" else False
    if latency_bound:
        # A few thousand flops per launch: the launch latency is the bound, no roofline applies.
        wk["bound"] = "latency"
        achieved = wk["flops"] / (dom_ms / 1e3) / 1e12
        peak = None
        unit = "TFLOP/s"
    elif dominant == "window_shift":
        # The window shift of a sliding-window cache: bytes of the rows it moves, read and written.
        wk["bound"] = "hbm"
        achieved = window_shift_bytes(case) / (dom_ms / 1e3) / 1e9
        peak = float(peaks["hbm_gbs"])
        peak_key = "hbm_gbs"
        unit = "GB/s"
    elif wk["bound"] == "hbm":
        achieved = wk["kv_bytes"] / (dom_ms / 1e3) / 1e9
        peak = float(peaks["hbm_gbs"])
        unit = "GB/s"
    elif dominant == "prefill_cuda_core":
        # fp32 attention on the CUDA cores: bound by fp32 FMA issue, not by the tensor pipe.
        wk["bound"] = "alu"
        achieved = wk["flops"] / (dom_ms / 1e3) / 1e12
        sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        peak = round(SM_COUNT * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12, 2)
        peak_key = f"fp32 FMA: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 flop x {sm_mhz:.0f} MHz"
        unit = "TFLOP/s"
    else:
        achieved = wk["flops"] / (dom_ms / 1e3) / 1e12
        peak = float(peaks["bf16_tflops"])
        unit = "TFLOP/s"
    traffic = recorded_traffic(name, kernel_src)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_baseline = oracle_sample(case, budget_s=args.cpu_budget)
        cpu_baseline.pop("seconds", None)
        cpu_baseline.pop("runs", None)

    if wk["bound"] == "latency":
        peak_source = "none (launch-latency bound)"
    elif wk["bound"] == "alu":
        peak_source = f"derived ({peak_key})"
    else:
        peak_source = f"{peaks_src} ({peak_key}, burst)"
    rec = {
        "value": round(value, 3),
        "unit": wk["unit"],
        "ms_per_step": round(ms, 5),
        "dtype": "f16" if sp.dtype == "f16" else "f32",
        "config": {"workload": name, "batch": sp.B, "seq_len": sp.S, "num_heads": sp.N,
                   "kv_num_heads": sp.Nkv, "head_size": sp.H, "capacity": sp.capacity,
                   "cache": (f"{sp.quant} int{sp.bits}" if sp.quant != "NONE" else (sp.cache_dtype or sp.dtype)),
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then read back)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "regime": "decode" if plan.regime == 1 else "prefill",
                   "split_len": int(plan.split_len), "max_splits": int(plan.max_splits),
                   "kernel_times": "CUDA events around each launch over a second pass of the same K steps"},
        "roofline": {"bound": wk["bound"], "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4) if peak else None, "traffic": traffic,
                     "peak_source": peak_source, "kernel": dominant, "kernel_ms": round(dom_ms, 5)},
        "kernels_ms": {k: round(sum(v) / len(v), 5) for k, v in per_kernel.items()},
        "e2e": {"value": round(e2e_value, 3), "unit": wk["unit"], "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(plan.launches) * args.steps,   # launches in the timed pass
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                   "samples": clocks["samples"]},
        "cpu_baseline": cpu_baseline,
    }
    op.close()
    del dev, pk, pv, out, ws, flush, flush_words, call, opt, call_e2e, staged, dev_stage, host_stage
    torch.cuda.empty_cache()
    return rec


# The workloads of the other configurations reported beside the headline one:
# the tiny fp32 prompt (launch latency), fp16 causal prefill (tensor cores),
# fp16 chunked prefill (tensor cores) and fp32 decode over an int8 cache (HBM).
CONFIG_WORKLOADS = ["prompt_f32_b1_s16", "prefill_f16_b4_s4096", "chunked_prefill_f16_b8_s512",
                    "decode_int8_f32_b32_c16384"]


def run_gpu_arm(args, world, rank, local) -> None:
    import torch

    torch.cuda.set_device(local)
    rec = measure_workload(args.workload, args, world, rank, local)
    extra = {}
    names = CONFIG_WORKLOADS if args.workloads == "configs" else \
        ([] if args.workloads == "none" else [w for w in args.workloads.split(",") if w])
    for w in names:
        if w != args.workload:
            extra[w] = measure_workload(w, args, world, rank, local)
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": rec["value"],
        "unit": rec["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": rec["dtype"],
        "data": "synthetic (seeded numpy, shapes and distributions of the workload)",
        "config": rec["config"],
        "roofline": rec["roofline"],
        "kernels_ms": rec["kernels_ms"],
        "e2e": rec["e2e"],
        "gpu_launches": rec["gpu_launches"] + sum(r["gpu_launches"] for r in extra.values()),
        "clocks": rec["clocks"],
        "cpu_baseline": rec["cpu_baseline"],
    }
    if extra:
        # Every other configuration, measured in this run the same way (its own clocks,
        # roofline of its dominant kernel, end-to-end value and oracle sample).
        line["workloads"] = extra
    print(json.dumps(line), flush=True)


def run_reference_arm(args, world, rank) -> None:
    if rank != 0:
        return
    case = generate(WORKLOADS[args.workload], seed=0)
    sp = case["spec"]
    for _ in range(args.warmup):
        oracle_sample(case, budget_s=0.0, max_runs=1)
    t0 = time.perf_counter()
    c0 = time.process_time()
    vals = []
    desc = None
    for _ in range(args.steps):
        r = oracle_sample(case, budget_s=0.0, max_runs=1)
        vals.append(r["seconds"])
        desc = r["sample"]
        units = r["value"] * r["seconds"]
    wall = time.perf_counter() - t0
    cores = max(1, round((time.process_time() - c0) / wall))
    ms = 1e3 * sum(vals) / len(vals)
    value = units / (ms / 1e3)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": work(case)["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded numpy, shapes and distributions of the workload)",
        "config": {"workload": args.workload, "batch": sp.B, "seq_len": sp.S, "num_heads": sp.N,
                   "kv_num_heads": sp.Nkv, "head_size": sp.H, "capacity": sp.capacity},
        "cpu_baseline": {"value": round(value, 6), "unit": work(case)["unit"], "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": work(case)["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=list(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load for clock sampling")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="configs",
                    help="other workloads measured in the same run and reported under 'workloads': "
                         "'configs' (the other configurations), 'none', or a comma-separated list")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least 3 untimed warm-up steps
    world, rank, local = dist_setup()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE {world}")
    if args.impl == "reference":
        run_reference_arm(args, world, rank)
    else:
        run_gpu_arm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
