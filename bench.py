#!/usr/bin/env python3
"""Benchmark of the fused LM-head loss on GB300.

One step = one fused cross-entropy forward + backward (lossk_ce_fwd_bwd:
validation, logit statistics, merge, token mean, d_hidden, d_weight) over one
synthetic batch of the Qwen3-0.6B head shape: n_tok=2048, d_model=1024,
vocab=151936, chunk 256, bf16, Zipf(1.1) targets.  Inputs are resident in
HBM when the timed region starts; the weight (311 MB) alone is larger than
L2, so no flush is needed between steps.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank takes its own batch (batch index = rank, same
weight) on its own GPU:
the ranks share no data, so N ranks are N independent replicas and the
whole-job value is N * n_tok / (max step time over ranks) ("weak").

Printed: one JSON line on rank 0.  The timed region runs with the library's
per-kernel tracing off; the per-kernel durations behind "roofline" and
"kernels" come from a second, traced loop of the same steps right after it.
Fractions of the bf16 tensor peak use the measured burst figure (the timed
regions here last well under a second); the sustained figure is reported
beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd tokens/s at Qwen3 shape; % of bf16 tensor peak"
WORKLOAD = "qwen3_0p6b_head"
# Which kernels' work counts as algorithmic (FLOPs per launch, in units of
# n*d*V multiply-adds x 2): statistics = one logit contraction; each backward
# pass = one logit contraction (recompute once) + its gradient contraction; the
# fused forward + d_hidden pass = one logit contraction + the d_hidden one.
ALGO_FLOPS_NDV = {"tc_stats": 2.0, "tc_rows": 4.0, "tc_cols": 4.0, "tc_fused": 4.0,
                  "fp_stats": 2.0, "fp_rows": 4.0, "fp_cols": 4.0}
HBM_KERNELS = {"from_logits", "validate", "merge_ce", "merge_distill", "reduce", "tokp_ce",
               "sum_splits", "tgt_logit", "merge_fused", "combine_dh", "teacher_stats",
               "distill_logits"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def args_parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the extra path measurements")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--paths-only", action="store_true",
                    help="time only the other rows of the path (distillation, CE from logits)")
    ap.add_argument("--path-tokens", type=int, default=None,
                    help="token count of the distillation workload in --paths-only mode")
    return ap.parse_args()


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(n_tok_per_rank, world, max_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * n_tok_per_rank / (max_ms / 1e3)


# ---- clocks -------------------------------------------------------------------

class Clocks:
    """nvidia-smi samples every 100 ms.  mark() brackets the timed region on the
    host clock; stop() keeps the samples taken inside it (all loaded samples if
    the region was shorter than the sampling interval, said in `window`)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.uuid = gpu_uuid
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def mark(self, begin):
        import datetime
        now = datetime.datetime.now()
        if begin:
            self.t0 = now
        else:
            self.t1 = now

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        rows = []
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9], ts))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[4] <= self.t1]
        window = "timed region"
        if not inside:
            # the timed region was shorter than the sampling interval: the samples
            # of the loaded window around it (untimed steps before and after)
            inside = [r for r in rows if r[2] > 0.3 * max(x[2] for x in rows)] or rows
            window = "loaded window around the timed region"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in inside),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(inside), "window": window, "power_w_max": max(r[2] for r in inside)}


# ---- traffic from the committed ncu summary -----------------------------------

def _code_only(text):
    """C/C++ source without comments and whitespace: a comment edit leaves the
    kernels, and so their recorded counters, unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch == '"' or ch == "'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    return "".join("".join(out).split())


# What builds the cluster passes and launches them: the kernel, the headers it
# includes, and the host side that encodes its tensor maps and launch shapes.
# The streaming and CTA-pair kernels are other translation units.
BWD_KERNEL_SRCS = ("output_projection_cross_gb300/csrc/k_bwp.cu",
                   "output_projection_cross_gb300/csrc/ptx.cuh",
                   "output_projection_cross_gb300/csrc/lossk_internal.h",
                   "output_projection_cross_gb300/csrc/lossk_abi.cu",
                   "include/lossk.h")


def kernel_src_sha(files=BWD_KERNEL_SRCS):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel)
    if not e or e.get("kernel_src_sha") != kernel_src_sha():
        return None
    return e.get("bytes_per_launch")


# ---- CPU baseline (the oracle, as it stands) --------------------------------------

def oracle_step(x, k, chunk):
    import oracle
    H, W, y = x["hidden"][:k], x["weight"], x["targets"][:k]
    m = None if x["mask"] is None else x["mask"][:k]
    oracle.ce_fwd(H, W, y, mask=m, chunk=min(chunk, k))
    oracle.ce_bwd(H, W, y, mask=m)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(x, chunk, seconds):
    """Oracle fwd+bwd on the first k tokens of the batch; k sized to ~`seconds`
    from a calibration run on 2 tokens per core (the oracle splits tokens
    across its threads, so fewer tokens would leave cores idle and overstate
    the time per token)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
    k0 = min(len(x["targets"]), 2 * cpu_cores())
    t0 = time.perf_counter()
    oracle_step(x, k0, chunk)
    tk = time.perf_counter() - t0
    k = int(max(k0, min(len(x["targets"]), k0 * seconds / max(tk, 1e-3))))
    t0 = time.perf_counter()
    oracle_step(x, k, chunk)
    dt = time.perf_counter() - t0
    return {"value": k / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"first {k} tokens of the batch (full d_model and vocab), fp64 fwd+bwd, "
                      f"{dt:.1f} s"}


# ---- our implementation -----------------------------------------------------------------

def WORKLOAD_OBJ():
    import lossk_inputs as li
    return li.WORKLOADS[WORKLOAD]


def run_ours(a, rank, world, local):
    import numpy as np
    import torch

    import lossk_inputs as li
    import output_projection_cross_gb300 as L

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = li.WORKLOADS[WORKLOAD]
    x = li.make(w, seed=0, batch=rank)
    H = torch.from_numpy(x["hidden"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["weight"]).to(dev).to(torch.bfloat16)
    y = torch.from_numpy(x["targets"]).to(dev)
    n, d, V = w.n_tok, w.d_model, w.vocab
    ws = L.workspace(L.lossk.KIND_CE_FWD_BWD, n, d, V, L.lossk.BF16, dev)
    out = dict(lse_out=torch.empty(n, device=dev), ce_out=torch.empty(n, device=dev),
               scalars_out=torch.empty(3, dtype=torch.float64, device=dev),
               d_hidden=torch.empty(n, d, device=dev), d_weight=torch.empty(V, d, device=dev))
    stream = torch.cuda.current_stream(dev)

    def step():
        L.lossk_ce_fwd_bwd(H, W, y, chunk=w.chunk, z_weight=w.z_weight, ws=ws, **out)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    assert L.lossk_device_status(ws) == 580

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = Clocks(uuid)
    # the sampler needs a moment to start: keep the GPU loaded with untimed
    # steps for ~0.4 s before the timed region and ~0.2 s after it
    clocks.start()
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 0.4:
        step()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = L.lossk_launch_count()
    clocks.mark(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    launches = L.lossk_launch_count() - launches0
    barrier(world)
    # the same steps again with per-kernel event pairs on each launch's stream:
    # the kernel durations (the timed region above runs without them)
    L.lossk_profile_read(reset=True)
    L.lossk_profile_enable(True)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(a.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    L.lossk_profile_enable(False)
    prof = L.lossk_profile_read(reset=True)
    ms_traced = t0.elapsed_time(t1) / a.steps
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 0.2:
        step()
        torch.cuda.synchronize()
    ck = clocks.stop()
    ms = e0.elapsed_time(e1) / a.steps
    ms_max = max_over_ranks(ms, world)
    assert L.lossk_device_status(ws) == 580

    pk = peaks()
    value = aggregate(n, world, ms_max)
    flops6 = 6.0 * n * d * V
    res = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_max,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded: hidden N(0,1), weight N(0,0.02), Zipf(1.1) targets)",
           "config": {"workload": WORKLOAD, "n_tok": n, "d_model": d, "vocab": V,
                      "chunk": w.chunk, "targets": w.targets,
                      "l2": "inputs larger than L2 (bf16 weight 311 MB > 126 MB L2); no flush",
                      "parallelism": f"{world} independent replica(s), one batch per rank"}}
    tflops = flops6 / (ms_max / 1e3) / 1e12
    res["tensor_peak"] = {"flops_per_step": flops6, "counted_as": "6*n*d*V",
                          "achieved_tflops": tflops, "peak_tflops": pk["bf16_tflops"],
                          "peak": f"bf16 burst ({pk['source']})",
                          "frac": tflops / pk["bf16_tflops"],
                          "frac_of_sustained": tflops / pk["bf16_tflops_sustained"],
                          "executed_flops_per_step": 8.0 * n * d * V,
                          "executed_frac": 8.0 * n * d * V / (ms_max / 1e3) / 1e12 / pk["bf16_tflops"]}
    # dominant kernel roofline: CUDA-event durations from the traced loop
    kern = {k: {"avg_ms": v[0] / v[1], "launches": v[1], "share": v[0] / (ms_traced * a.steps)}
            for k, v in prof.items()}
    dom = max(prof, key=lambda k: prof[k][0])
    avg = prof[dom][0] / prof[dom][1]
    if dom in ALGO_FLOPS_NDV:
        fl = ALGO_FLOPS_NDV[dom] * n * d * V
        ach = fl / (avg / 1e3) / 1e12
        peak = pk["bf16_tflops"]
        res["roofline"] = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak,
                           "unit": "TFLOP/s", "frac": ach / peak,
                           "peak_kind": f"bf16 burst, {pk['source']}",
                           "frac_of_sustained": ach / pk["bf16_tflops_sustained"],
                           "algorithmic_per_launch": fl,
                           "duration": f"average of {prof[dom][1]} launches, CUDA events on the launching "
                                       f"stream, traced loop of {a.steps} steps after the timed region",
                           "traffic": ncu_traffic(dom)}
    res["kernels"] = kern
    res["kernels_loop_ms_per_step"] = ms_traced
    res["gpu_launches"] = launches
    res["clocks"] = ck

    if not a.no_e2e:
        res["e2e"] = e2e(a, x, H, W, y, out, step, stream, n, world)
    if not a.quick and rank == 0:
        res["paths"] = extra_paths(L, dev, pk)
    if rank == 0 and world == 1 and not a.no_cpu:
        res["cpu_baseline"] = cpu_baseline(x, w.chunk, a.cpu_seconds)
    return res


def e2e(a, x, H, W, y, out, step, stream, n, world):
    """The same step through the public call with host buffers.  Every timed
    step copies its inputs (hidden, weight, targets) from pinned host memory to
    the device and its outputs (lse, ce, scalars, d_hidden, d_weight) back to
    pinned host memory.  The copies are pipelined the way a training loop feeds
    a device: step i+1's inputs travel on a copy stream while step i computes,
    and step i's gradients travel back on another while step i+1 computes.
    Device buffers are doubled for that; the timed region runs from the first
    input copy to the last output copy."""
    import numpy as np
    import torch

    import output_projection_cross_gb300 as L

    w = WORKLOAD_OBJ()
    dev = H.device
    hH = torch.from_numpy(x["hidden"]).to(torch.bfloat16).pin_memory()
    hW = torch.from_numpy(x["weight"]).to(torch.bfloat16).pin_memory()
    hy = torch.from_numpy(x["targets"]).pin_memory()
    bi = hH.numel() * 2 + hW.numel() * 2 + hy.numel() * 8
    ins = [(H, W, y), (torch.empty_like(H), torch.empty_like(W), torch.empty_like(y))]
    outs = [out, {k: torch.empty_like(v) for k, v in out.items()}]
    o_h = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()} for _ in range(2)]
    bo = sum(v.numel() * v.element_size() for v in o_h[0].values())
    ws = L.workspace(L.lossk.KIND_CE_FWD_BWD, n, H.shape[1], W.shape[0], L.lossk.BF16, dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(k_steps, timed):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for e in comp_done + out_done:
            e.record(stream)
        with torch.cuda.stream(s_in):
            if timed:
                e0.record(s_in)
            hb, wb, yb = ins[0]
            hb.copy_(hH, non_blocking=True)
            wb.copy_(hW, non_blocking=True)
            yb.copy_(hy, non_blocking=True)
            in_done[0].record(s_in)
        for i in range(k_steps):
            b = i % 2
            if i + 1 < k_steps:
                nb = (i + 1) % 2
                with torch.cuda.stream(s_in):
                    s_in.wait_event(comp_done[nb])          # step i-1 no longer reads buffer nb
                    hb, wb, yb = ins[nb]
                    hb.copy_(hH, non_blocking=True)
                    wb.copy_(hW, non_blocking=True)
                    yb.copy_(hy, non_blocking=True)
                    in_done[nb].record(s_in)
            stream.wait_event(in_done[b])
            stream.wait_event(out_done[b])                  # step i-2's outputs have left buffer b
            hb, wb, yb = ins[b]
            L.lossk_ce_fwd_bwd(hb, wb, yb, chunk=w.chunk, z_weight=w.z_weight, ws=ws, **outs[b])
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for k, v in outs[b].items():
                    o_h[b][k].copy_(v, non_blocking=True)
                out_done[b].record(s_out)
        stream.wait_event(out_done[(k_steps - 1) % 2])
        if timed:
            e1.record(stream)
        torch.cuda.synchronize()
        return e0, e1

    run(2, False)
    barrier(world)
    k_e2e = max(3, min(a.steps, 20))
    e0, e1 = run(k_e2e, True)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / k_e2e, world)
    # the results that came back match the device-resident step's
    assert np.array_equal(o_h[(k_e2e - 1) % 2]["scalars_out"].numpy(), out["scalars_out"].cpu().numpy())

    # The host link alone (untimed for the metric): the step's copies in both
    # directions at once, no compute -- the floor the pipelined step can reach.
    def copies():
        ev = torch.cuda.Event()
        ev.record(stream)
        s_in.wait_event(ev)
        s_out.wait_event(ev)
        with torch.cuda.stream(s_in):
            hb, wb, yb = ins[0]
            hb.copy_(hH, non_blocking=True)
            wb.copy_(hW, non_blocking=True)
            yb.copy_(hy, non_blocking=True)
        with torch.cuda.stream(s_out):
            for k, v in outs[1].items():
                o_h[1][k].copy_(v, non_blocking=True)
        for s in (s_in, s_out):
            e = torch.cuda.Event()
            e.record(s)
            stream.wait_event(e)
    floor_ms = _time(copies, 3, warm=1)
    return {"value": aggregate(n, world, e2e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
            "overlap": "next step's inputs and previous step's outputs copied during the current step",
            "copy_floor_ms": floor_ms,
            "copy_floor": "the same copies in both directions at once with no compute (host link bound)"}


def _time(fn, reps, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _time_traced(L, fn, reps, warm=2):
    """(ms per call untraced, {kernel: average ms} from a second, traced run)."""
    ms = _time(fn, reps, warm)
    L.lossk_profile_read(reset=True)
    L.lossk_profile_enable(True)
    _time(fn, reps, 0)
    L.lossk_profile_enable(False)
    prof = L.lossk_profile_read(reset=True)
    return ms, {k: v[0] / v[1] for k, v in prof.items()}


def ce_step_path(L, dev, pk, wl, reps=5):
    """lossk_ce_fwd_bwd on a workload's own recipe (mask, z weight), bf16."""
    import torch

    import lossk_inputs as li
    w = li.WORKLOADS[wl]
    x = li.make(w, seed=0)
    n, d, V = w.n_tok, w.d_model, w.vocab
    H = torch.from_numpy(x["hidden"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["weight"]).to(dev).to(torch.bfloat16)
    y = torch.from_numpy(x["targets"]).to(dev)
    m = None if x["mask"] is None else torch.from_numpy(x["mask"]).to(dev)
    del x
    ws = L.workspace(L.lossk.KIND_CE_FWD_BWD, n, d, V, L.lossk.BF16, dev)
    out = dict(lse_out=torch.empty(n, device=dev), ce_out=torch.empty(n, device=dev),
               scalars_out=torch.empty(3, dtype=torch.float64, device=dev),
               d_hidden=torch.empty(n, d, device=dev), d_weight=torch.empty(V, d, device=dev))

    def fn():
        L.lossk_ce_fwd_bwd(H, W, y, loss_mask=m, chunk=w.chunk, z_weight=w.z_weight, ws=ws, **out)
    ms, kms = _time_traced(L, fn, reps)
    fl6 = 6.0 * n * d * V
    dom = max((k for k in kms if k in ALGO_FLOPS_NDV), key=lambda k: kms[k])
    r = {"workload": wl, "ms": ms, "tokens_per_s": n / (ms / 1e3), "flops_counted": fl6,
         "counted_as": "6*n*d*V", "tensor_frac": fl6 / (ms / 1e3) / 1e12 / pk["bf16_tflops"],
         "peak": "bf16 burst", "kernels_ms": kms,
         "dominant": {"kernel": dom, "avg_ms": kms[dom],
                      "frac": ALGO_FLOPS_NDV[dom] * n * d * V / (kms[dom] / 1e3) / 1e12 / pk["bf16_tflops"]}}
    del H, W, y, m, ws, out
    torch.cuda.empty_cache()
    return r


def extra_paths(L, dev, pk, n_tok=None):
    """The other rows of the hot path, timed the same way: distillation at
    n=4096, d=2048, V=151936 (T=2, 10% masked, z 1e-4; n_tok overrides the
    token count) and cross-entropy from materialised bf16 logits at the Qwen3
    head shape (HBM stream)."""
    import dataclasses

    import torch

    import lossk_inputs as li
    res = {}
    w = li.WORKLOADS["distill_z_4096x2048"]
    if n_tok is not None:
        w = dataclasses.replace(w, n_tok=n_tok)
    x = li.make(w, seed=0)
    H = torch.from_numpy(x["hidden"]).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(x["weight"]).to(dev).to(torch.bfloat16)
    T = torch.from_numpy(x["teacher"]).to(dev).to(torch.bfloat16)
    m = torch.from_numpy(x["mask"]).to(dev)
    del x
    ws = L.workspace(L.lossk.KIND_DISTILL, w.n_tok, w.d_model, w.vocab, 1, dev)
    bufs = dict(d_hidden=torch.empty(w.n_tok, w.d_model, device=dev),
                d_weight=torch.empty(w.vocab, w.d_model, device=dev))
    for direction in w.directions:
        def fn():
            L.lossk_distill_fwd_bwd(H, W, T, direction, temperature=w.temperature, loss_mask=m,
                                    chunk=w.chunk, z_weight=w.z_weight, ws=ws, **bufs)
        ms, kms = _time_traced(L, fn, 3)
        fl = 6.0 * w.n_tok * w.d_model * w.vocab
        # the teacher stream on its own (the teacher statistics kernel reads
        # every teacher logit once): its HBM roofline
        tbytes = w.n_tok * w.vocab * 2
        tk = kms.get("teacher_stats")
        res[f"distill_{direction}"] = {
            "workload": w.name, "ms": ms, "tokens_per_s": w.n_tok / (ms / 1e3),
            "tensor_frac_6ndV": fl / (ms / 1e3) / 1e12 / pk["bf16_tflops"], "peak": "bf16 burst",
            "kernels_ms": kms,
            "teacher_stream": None if tk is None else {
                "kernel": "teacher_stats", "algorithmic_bytes": tbytes, "kernel_ms": tk,
                "achieved_gbs": tbytes / (tk / 1e3) / 1e9,
                "frac_hbm": tbytes / (tk / 1e3) / 1e9 / pk["hbm_gbs"]}}
    del H, W, T, bufs
    torch.cuda.empty_cache()
    # CE from materialised logits (HBM-bound): read 622 MB bf16, write 622 MB grad
    n, V = 2048, 151936
    g = torch.Generator(device=dev).manual_seed(0)
    X = torch.randn(n, V, device=dev, generator=g).to(torch.bfloat16)
    y = torch.randint(0, V, (n,), device=dev, generator=g)
    grad = torch.empty_like(X)
    ws = L.workspace(L.lossk.KIND_FROM_LOGITS, n, 1, V, 1, dev)
    for want in (False, True):
        def fn():
            L.lossk_ce_from_logits(X, y, grad_logits=grad if want else None, want_grad=want, ws=ws)
        ms, kall = _time_traced(L, fn, 5)
        kms = kall["from_logits"]
        nbytes = X.numel() * 2 * (2 if want else 1)
        res["from_logits" + ("_grad" if want else "")] = {
            "workload": "logits bf16 [2048][151936]", "ms": ms,
            "kernel_ms": kms, "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / (kms / 1e3) / 1e9,
            "frac_hbm": nbytes / (kms / 1e3) / 1e9 / pk["hbm_gbs"]}
    # the label loss's other entry points at the Qwen3 head shape: the forward
    # alone (CTA-pair statistics), the backward alone (both separate passes), and
    # the training step with fp16 inputs (the separate passes: the single-pass
    # forward + d_hidden needs bf16's range)
    del X, grad
    torch.cuda.empty_cache()
    wq = li.WORKLOADS["qwen3_0p6b_head"]
    xq = li.make(wq, seed=0)
    nq, dq, Vq = wq.n_tok, wq.d_model, wq.vocab
    yq = torch.from_numpy(xq["targets"]).to(dev)
    fl6 = 6.0 * nq * dq * Vq
    for dt_name, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        Hq = torch.from_numpy(li.round_to(xq["hidden"], dt_name)).to(dev).to(tdt)
        Wq = torch.from_numpy(li.round_to(xq["weight"], dt_name)).to(dev).to(tdt)
        code = L.lossk.BF16 if dt_name == "bf16" else L.lossk.F16
        dH = torch.empty(nq, dq, device=dev)
        dW = torch.empty(Vq, dq, device=dev)
        lse = torch.empty(nq, device=dev)
        calls = {}
        if dt_name == "bf16":
            wsf = L.workspace(L.lossk.KIND_CE_FWD, nq, dq, Vq, code, dev)
            wsb = L.workspace(L.lossk.KIND_CE_BWD, nq, dq, Vq, code, dev)
            L.lossk_ce_fwd(Hq, Wq, yq, chunk=wq.chunk, lse_out=lse, ws=wsf)
            calls["ce_fwd_only"] = (lambda: L.lossk_ce_fwd(Hq, Wq, yq, chunk=wq.chunk, lse_out=lse, ws=wsf), 2.0)
            calls["ce_bwd_only"] = (lambda: L.lossk_ce_bwd(Hq, Wq, yq, lse, d_hidden=dH, d_weight=dW, ws=wsb), 4.0)
        else:
            wss = L.workspace(L.lossk.KIND_CE_FWD_BWD, nq, dq, Vq, code, dev)
            calls["ce_fwd_bwd_f16"] = (lambda: L.lossk_ce_fwd_bwd(Hq, Wq, yq, chunk=wq.chunk, d_hidden=dH,
                                                                  d_weight=dW, ws=wss), 6.0)
        for name, (fn, units) in calls.items():
            ms, kms = _time_traced(L, fn, 5)
            fl = units / 6.0 * fl6
            res[name] = {"workload": f"{wq.name} ({dt_name})", "ms": ms, "tokens_per_s": nq / (ms / 1e3),
                         "flops_counted": fl, "counted_as": f"{int(units)}*n*d*V",
                         "tensor_frac": fl / (ms / 1e3) / 1e12 / pk["bf16_tflops"], "peak": "bf16 burst",
                         "kernels_ms": kms}
        del Hq, Wq, dH, dW
        torch.cuda.empty_cache()
    X = torch.randn(n, V, device=dev, generator=g).to(torch.bfloat16)
    grad = torch.empty_like(X)
    # distillation from given student logits (HBM stream): read the student and
    # teacher logits once, write grad_logits once
    T = (torch.randn(n, V, device=dev, generator=g) * 3).to(torch.bfloat16)
    ws = L.workspace(L.lossk.KIND_FROM_LOGITS, n, 1, V, 1, dev)
    for want in (False, True):
        def fn():
            L.lossk_distill_from_logits(X, T, "fkl", temperature=2.0, z_weight=1e-4, want_grad=want,
                                        grad_logits=grad if want else None, ws=ws)
        ms, kall = _time_traced(L, fn, 5)
        kms = kall["distill_logits"]
        nbytes = X.numel() * 2 * (3 if want else 2)
        res["distill_from_logits" + ("_grad" if want else "")] = {
            "workload": "student and teacher logits bf16 [2048][151936], forward KL, T 2",
            "ms": ms, "kernel_ms": kms, "algorithmic_bytes": nbytes,
            "achieved_gbs": nbytes / (kms / 1e3) / 1e9,
            "frac_hbm": nbytes / (kms / 1e3) / 1e9 / pk["hbm_gbs"]}
    del X, T, grad, ws
    torch.cuda.empty_cache()
    # the label loss's two other configurations, at their own recipes
    res["ce_512x1024x32000"] = ce_step_path(L, dev, pk, "ce_512x1024x32000", reps=20)
    res["ce_z_8192x4096x128256"] = ce_step_path(L, dev, pk, "ce_z_8192x4096x128256", reps=3)
    return res


# ---- the reference arm: the oracle, as it stands ------------------------------------

def run_reference(a, rank, world):
    if rank != 0:
        return None
    import lossk_inputs as li
    w = li.WORKLOADS[WORKLOAD]
    x = li.make(w, seed=0)
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
    # size one step's sample so that warmup + steps fit in about three minutes:
    # a first call pays the oracle's one-time start-up (seconds), so the
    # calibration is the second call, on 2 tokens per core (the oracle splits
    # tokens across its threads)
    k0 = min(w.n_tok, 2 * cpu_cores())
    oracle_step(x, k0, w.chunk)
    t0 = time.perf_counter()
    oracle_step(x, k0, w.chunk)
    tk = time.perf_counter() - t0
    per_step = min(8.0, 170.0 / max(1, a.steps + a.warmup))
    k = int(max(1, min(w.n_tok, k0 * per_step / max(tk, 1e-3))))
    for _ in range(a.warmup):
        oracle_step(x, k, w.chunk)
    t0 = time.perf_counter()
    for _ in range(a.steps):
        oracle_step(x, k, w.chunk)
    dt = (time.perf_counter() - t0) / a.steps
    v = k / dt
    sample = f"first {k} tokens of the batch per step (full d_model and vocab), fp64 fwd+bwd"
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_tok": w.n_tok, "d_model": w.d_model,
                       "vocab": w.vocab, "chunk": w.chunk, "targets": w.targets},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    a = args_parse()
    if a.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit at once
        rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(a, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, local = dist_init()
    if a.paths_only:
        import torch
        import output_projection_cross_gb300 as L
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        if rank == 0:
            print(json.dumps({"paths": extra_paths(L, dev, peaks(), a.path_tokens)}), flush=True)
        return
    res = run_ours(a, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
