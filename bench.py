#!/usr/bin/env python3
"""Benchmark of the GB300 dense GEMM / GEMV / expert-ID matmul hot path.

One step = one pass over the whole hot path, the five synthetic workloads
(seed 0) each called once through the C ABI, in this order:
  C5  matmul_id GroupedPrefill  m=4096 E=128 top_k=8 (Zipf 1.1) k=4096 n=1536 bf16 W
  C3  batched GEMM f16          4 x 4096 x 4096 x 4096 (B stored [n,k])
  C2  decode GEMV f16           1 x 11008 x 4096 (W stored [n,k])
  C4  matmul_id Direct          m=4 E=64 top_k=8 k=2048 n=1408 bf16 W
  C1  f32 GEMM                  64 x 64 x 128
Every call starts with its inputs evicted from L2 by the calls before it
(C5 streams 1.9 GB, C3 moves 0.4 GB).  The two large writers come first:
the dirty lines of C5's 201 MB output are written back while C3 computes
(C3 is tensor-bound and leaves HBM mostly idle) rather than during the
reads of an HBM-bound decode call.
Metric: "% of GB300 roofline" = sum over the calls of their roofline time
(max(algorithmic flops / tensor or FFMA peak, algorithmic bytes / HBM
peak), peaks from MEASURED_PEAKS.json) divided by the measured step time.
With N GPUs (torchrun) every rank runs the same step (replicas: the path has
no exchange step); value = N * sum(roofline) / max-over-ranks step time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--only c1,c2,...] [--no-e2e] [--no-cpu-baseline] [--no-steady] [--no-options]
       [--no-sweeps] [--sweep crossover|skinny|dtypes|ffma]
Roofline peaks: the measured HBM copy rate and the burst bf16 tensor rate
(the timed region lasts tens of milliseconds).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemv_moe_expert_gb300 import synth  # noqa: E402

ORDER = ["c5", "c3", "c2", "c4", "c1"]
NAMES = {"c1": "c1_f32_gemm", "c2": "c2_f16_gemv", "c3": "c3_f16_gemm",
         "c4": "c4_moe_direct", "c5": "c5_moe_grouped"}
METRIC = "GEMM TFLOP/s and GEMV/matmul_id GB/s, as % of GB300 roofline"
UNIT = "% of GB300 roofline (sum of per-call roofline times / step time)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def ffma_peak_tflops(sm_mhz: float = 2070.0, sms: int = 152) -> float:
    # 128 FP32 FMA lanes per SM per clock, 2 flops per FMA
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


# ---------------------------------------------------------------------------
# per-workload algorithmic work
# ---------------------------------------------------------------------------

def work_of(key: str, w) -> dict:
    if key in ("c1", "c2", "c3"):
        size = synth.ITEMSIZE[w.dtype]
        flops = 2 * w.batch * w.m * w.n * w.k
        bytes_ = (w.a.size + w.b.size + w.batch * w.m * w.n) * size
        bound = "tensor" if key == "c3" else ("hbm" if key == "c2" else "ffma")
        return {"flops": flops, "bytes": bytes_, "bound": bound}
    c = w
    wsize = synth.ITEMSIZE[c.wdtype]
    expert_bytes = c.n * c.k * wsize
    distinct = len(np.unique(c.ids.reshape(-1)[c.ids.reshape(-1) < c.n_experts]))
    flops = 2 * c.m * c.top_k * c.n * c.k
    if key == "c4":
        # the distinct experts of the call are read once
        bytes_ = distinct * expert_bytes + c.x.nbytes + c.ids.nbytes + c.m * c.top_k * c.n * 4
        return {"flops": flops, "bytes": bytes_, "bound": "hbm", "distinct_experts": distinct}
    bytes_ = c.n_experts * expert_bytes + c.x.nbytes + c.ids.nbytes + c.m * c.top_k * c.n * 4
    return {"flops": flops, "bytes": bytes_, "bound": "hbm+tensor", "distinct_experts": distinct}


def roofline_seconds(wk: dict, peaks: dict, tensor_peak_tf: float) -> float:
    t_bytes = wk["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if wk["bound"] == "ffma":
        t_flops = wk["flops"] / (ffma_peak_tflops() * 1e12)
    else:
        t_flops = wk["flops"] / (tensor_peak_tf * 1e12)
    return max(t_bytes, t_flops)


# ---------------------------------------------------------------------------
# CPU oracle baseline (the oracle as it stands, on the host cores)
# ---------------------------------------------------------------------------

# Calls the oracle finishes on every output in well under a second; the two
# large calls (2.7e11 and 2.1e11 multiply-adds) are timed on a sample of their
# outputs and extrapolated by output count.
FULL_CPU_KEYS = ("c1", "c2", "c4")
CPU_SAMPLE = {"c3": 1572864, "c5": 1572864}  # cpu_baseline leg of our arm (~10-15 s on 16 cores)
REF_SAMPLE = {"c3": 32768, "c5": 32768}     # each step of the reference arm


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the record beside the core count."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_call_seconds(key: str, w, outputs: int | None, threads: int) -> tuple[float, int, int]:
    """Time the oracle on one call: every output when `outputs` is None, else
    on that many sampled outputs.  Returns (seconds, outputs timed, outputs
    of the call)."""
    import oracle
    rng = np.random.default_rng(123)
    if key in ("c1", "c2", "c3"):
        total = w.batch * w.m * w.n
        cnt = total if outputs is None else min(outputs, total)
        idx = rng.choice(total, cnt, replace=False).astype(np.int64) if cnt < total else None
        t0 = time.perf_counter()
        oracle.gemm(w.dtype, w.batch, w.m, w.n, w.k, w.ta, w.tb, w.a.reshape(-1), w.lda,
                    w.stride_a, w.b.reshape(-1), w.ldb, w.stride_b, idx=idx, nthreads=threads)
        return time.perf_counter() - t0, cnt, total
    c = w
    total = c.m * c.top_k * c.n
    cnt = total if outputs is None else min(outputs, total)
    idx = rng.choice(total, cnt, replace=False).astype(np.int64) if cnt < total else None
    t0 = time.perf_counter()
    oracle.matmul_id(c.wdtype, c.m, c.n, c.k, c.top_k, c.n_experts, c.expert_stride_bytes,
                     c.input_layout, c.w, c.x, c.ids, idx=idx, nthreads=threads)
    if c.route == 1:
        oracle.map_distinct(c.m, c.top_k, c.n_experts, c.ids)
    return time.perf_counter() - t0, cnt, total


def cpu_step(workloads: dict, keys, sample: dict, scale: float = 1.0) -> dict:
    """One pass of the oracle over the step's calls: every output of the small
    calls, a sample of the large ones (extrapolated by output count)."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    calls, measured, est = {}, 0.0, 0.0
    for key in keys:
        n_out = None if key in FULL_CPU_KEYS else max(1, int(sample[key] * scale))
        secs, cnt, total = oracle_call_seconds(key, workloads[key], n_out, threads)
        calls[key] = {"seconds": secs, "outputs_timed": cnt, "outputs": total,
                      "extrapolated": cnt < total, "est_seconds": secs * total / cnt}
        measured += secs
        est += secs * total / cnt
    desc = ", ".join(f"{k}: {v['outputs_timed']}/{v['outputs']} outputs" +
                     (" (extrapolated)" if v["extrapolated"] else "") for k, v in calls.items())
    return {"cores": threads, "cpu_model": cpu_model(), "measured_seconds": measured,
            "est_step_seconds": est, "calls": calls, "sample": desc}


def cpu_baseline(workloads: dict, roof_total: float, scale: float = 1.0) -> dict:
    cb = cpu_step(workloads, [k for k in ORDER if k in workloads], CPU_SAMPLE, scale)
    est_total = cb["est_step_seconds"]
    return {"value": 100.0 * roof_total / est_total, "unit": UNIT, "cores": cb["cores"],
            "cpu_model": cb["cpu_model"], "kind": "oracle",
            "sample": cb["sample"] + f"; {cb['measured_seconds']:.1f} s measured, full step "
                                     f"{est_total:.1f} s with the sampled calls extrapolated",
            "measured_seconds": cb["measured_seconds"], "est_step_seconds": est_total,
            "calls": cb["calls"]}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

class Problem:
    """Device buffers and the call of one workload."""

    def __init__(self, key, w, torch, gb):
        self.key, self.w = key, w
        self.torch, self.gb = torch, gb
        dev = torch.device("cuda")

        def up(arr):
            return torch.from_numpy(np.ascontiguousarray(arr).reshape(-1).view(np.uint8).copy()).to(dev)

        self.host_inputs = []
        if key in ("c1", "c2", "c3"):
            self.a, self.b = up(w.a), up(w.b)
            self.c = torch.empty(w.batch * w.m * w.n * synth.ITEMSIZE[w.dtype], dtype=torch.uint8,
                                 device=dev)
            self.host_inputs = [w.a, w.b]
            self.outputs = [self.c]
            self.launches = 1
        else:
            c = w
            self.wt, self.x, self.ids = up(c.w), up(c.x), up(c.ids)
            self.params = gb.make_params(c.m, c.n, c.k, c.top_k, c.n_experts, c.expert_stride_bytes,
                                         c.input_layout, c.multiplicity, c.route)
            st, cap = gb.gbmm_matmul_id_capability(c.wdtype, self.params)
            gb.check(st)
            self.cap = cap
            self.out = torch.empty(cap.required_output_bytes, dtype=torch.uint8, device=dev)
            self.scratch = None
            if c.route == 1:
                self.counts = torch.empty(cap.expert_counts_bytes, dtype=torch.uint8, device=dev)
                self.rows = torch.empty(cap.routed_rows_bytes, dtype=torch.uint8, device=dev)
                self.scratch = gb.make_scratch(self.counts, cap.expert_counts_bytes, self.rows,
                                               cap.routed_rows_bytes, c.n_experts, c.m)
            self.host_inputs = [c.w, c.x, c.ids]
            self.outputs = [self.out]
            self.launches = 2 if c.route == 1 else 1

    def device_inputs(self):
        if self.key in ("c1", "c2", "c3"):
            return [self.a, self.b]
        return [self.wt, self.x, self.ids]

    def call(self, stream, inputs=None):
        """One call on `stream`; `inputs` (same order as device_inputs()) swaps
        in another copy of the input buffers."""
        gb, w = self.gb, self.w
        ins = inputs if inputs is not None else self.device_inputs()
        if self.key in ("c1", "c2", "c3"):
            fn = gb.gbmm_gemv if self.key == "c2" else gb.gbmm_gemm
            st = fn(w.dtype, w.batch, w.m, w.n, w.k, w.ta, w.tb, ins[0], 0, w.lda, w.stride_a,
                    ins[1], 0, w.ldb, w.stride_b, self.c, 0, w.ldc, w.stride_c, stream)
        else:
            c = w
            st, _ = gb.gbmm_matmul_id(self.params, c.wdtype, ins[0], c.w.nbytes, ins[1],
                                      c.x.nbytes, ins[2], c.ids.nbytes, self.out,
                                      self.cap.required_output_bytes, self.scratch, stream)
        if st != gb.GBMM_OK:
            raise RuntimeError(f"{self.key}: {gb.gbmm_status_string(st)}: {gb.gbmm_last_error()}")


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks of the default process group (the value
    itself without one).  Works with gloo (CPU tensors) and nccl (device)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_value(roof_total_s: float, world: int, ms_per_step: float) -> float:
    """Whole-job % of one GB300's roofline: every rank runs one full step."""
    return 100.0 * world * roof_total_s / (ms_per_step / 1e3)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_ours(args) -> None:
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from gemv_moe_expert_gb300 import binding as gb
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()

    keys = [k for k in ORDER if k in args.only]
    peaks, peak_src = load_peaks()
    # the timed region is a few tens of milliseconds: the burst tensor rate
    tensor_peak = peaks["bf16_tflops"]
    workloads = {k: synth.workload(NAMES[k]) for k in keys}
    works = {k: work_of(k, workloads[k]) for k in keys}
    roof = {k: roofline_seconds(works[k], peaks, tensor_peak) for k in keys}
    roof_total = sum(roof.values())

    probs = {k: Problem(k, workloads[k], torch, gb) for k in keys}
    stream = torch.cuda.Stream()
    sptr = int(stream.cuda_stream)
    n_launch = sum(p.launches for p in probs.values())

    def step(events=None, around=None):
        # events[i] before call i and events[-1] after the last one; with
        # `around`, only events[0] / events[1] around that call
        for i, k in enumerate(keys):
            if events is not None and (around is None or k == around):
                events[0 if around else i].record(stream)
            probs[k].call(sptr)
            if events is not None and k == around:
                events[1].record(stream)
        if events is not None and around is None:
            events[len(keys)].record(stream)

    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # per-call split: an instrumented pass with an event between every two
    # launches (each event costs a few microseconds of the step, so the
    # timed steps below carry events around the dominant call only)
    split_steps = max(3, min(args.steps, 10))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(keys) + 1)] for _ in range(split_steps)]
    for s in range(split_steps):
        step(ev[s])
    torch.cuda.synchronize()
    per_call = {k: sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(split_steps)) / split_steps
                for i, k in enumerate(keys)}
    dom = max(keys, key=lambda k: per_call[k])

    # the timed steps: the whole hot path back to back, the dominant call's
    # launches bracketed by events on the launching stream
    dev_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    gb.gbmm_test_reset_launch_count()
    t_wall = time.perf_counter()
    start.record(stream)
    for s in range(args.steps):
        step(dev_ev[s], around=dom)
    end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    launches = gb.gbmm_test_launch_count()
    if world > 1:
        dist.barrier()
    time.sleep(0.1)
    clk = clocks.stop()
    elapsed_ms = start.elapsed_time(end)
    dom_ms_live = sum(e[0].elapsed_time(e[1]) for e in dev_ev) / args.steps
    # per-step times at no extra cost: every step records one event at the
    # same place (just before the dominant call), so consecutive ones are one
    # step apart
    step_ms = [dev_ev[s][0].elapsed_time(dev_ev[s + 1][0]) for s in range(args.steps - 1)]
    if keys and keys[0] == dom:
        step_ms.append(dev_ev[args.steps - 1][0].elapsed_time(end))
    per_call_split = dict(per_call)
    per_call[dom] = dom_ms_live

    elapsed_ms = max_over_ranks(elapsed_ms, device="cuda")
    ms_per_step = elapsed_ms / args.steps
    value = step_value(roof_total, world, ms_per_step)

    # ---- end to end: pinned host inputs in, results out, every step ----
    # Every step copies each call's inputs from pinned host memory and reads
    # each call's output back.  The copies run on their own streams so that
    # they overlap the other calls' kernels the way a serving loop would: the
    # inputs of call i+1 stream in while call i computes, and the output of
    # call i streams out meanwhile.  Across steps, a call's input buffers are
    # refilled only after its previous kernels are done, and its output is
    # overwritten only after its previous read-back is done.
    e2e = None
    if not args.no_e2e:
        ins, outs = {}, {}
        for k in keys:
            p = probs[k]
            ins[k] = []
            for host, dev_t in zip(p.host_inputs, p.device_inputs()):
                h = torch.from_numpy(np.ascontiguousarray(host).reshape(-1).view(np.uint8).copy())
                ins[k].append((dev_t, h.pin_memory()))
            outs[k] = [(torch.empty(dev_t.numel(), dtype=torch.uint8).pin_memory(), dev_t) for dev_t in p.outputs]
        h2d = sum(h.numel() for k in keys for _, h in ins[k])
        d2h = sum(h.numel() for k in keys for h, _ in outs[k])
        e2e_steps = max(1, min(args.steps, 5))
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        done_ev = {k: None for k in keys}   # kernels of call k finished (previous step)
        read_ev = {k: None for k in keys}   # output of call k read back (previous step)

        def e2e_step(copy_events=None):
            for i, k in enumerate(keys):
                with torch.cuda.stream(s_in):
                    if done_ev[k] is not None:
                        s_in.wait_event(done_ev[k])
                    for dev_t, h in ins[k]:
                        dev_t.copy_(h, non_blocking=True)
                    landed = torch.cuda.Event()
                    landed.record(s_in)
                    if copy_events is not None and i == len(keys) - 1:
                        copy_events[1].record(s_in)
                stream.wait_event(landed)
                if read_ev[k] is not None:
                    stream.wait_event(read_ev[k])
                probs[k].call(sptr)
                done = torch.cuda.Event()
                done.record(stream)
                done_ev[k] = done
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done)
                    for h, dev_t in outs[k]:
                        h.copy_(dev_t, non_blocking=True)
                    rd = torch.cuda.Event()
                    rd.record(s_out)
                    read_ev[k] = rd
            # the step ends when every read-back has landed
            for k in keys:
                stream.wait_event(read_ev[k])

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        s_in.wait_event(s0)
        s_out.wait_event(s0)
        with torch.cuda.stream(s_in):
            c0.record(s_in)
        for j in range(e2e_steps):
            e2e_step([None, c1] if j == e2e_steps - 1 else None)
        s1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(s0.elapsed_time(s1) / e2e_steps, device="cuda")
        copy_ms = c0.elapsed_time(c1) / e2e_steps
        e2e = {"value": step_value(roof_total, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "steps": e2e_steps,
               "h2d_stream_ms_per_step": copy_ms,
               "note": "inputs copied from pinned host memory on a copy stream, outputs read back on "
                       "another, overlapped with the other calls' kernels; bound by the host link"}

    # side measurement (not part of the step): the grouped workload with the
    # opt-in single bf16 rounding of the activations, same buffers and order
    single = None
    if "c5" in probs and not args.no_options:
        pc = probs["c5"]
        default_precision = pc.params.activation_precision
        pc.params.activation_precision = gb.ACT_BF16
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        for _ in range(2):
            pc.call(sptr)
        times = []
        for _ in range(max(3, args.steps // 2)):
            with torch.cuda.stream(stream):
                flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pc.call(sptr)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        pc.params.activation_precision = default_precision
        del flush
        ms = statistics.median(times)
        single = {"ms": ms, "roofline_ms": roof["c5"] * 1e3,
                  "frac_of_roofline": roof["c5"] * 1e3 / ms,
                  "note": "matmul_id GroupedPrefill with activation_precision=bf16 (opt-in: one "
                          "bf16 rounding of the activations, half the tensor work; default splits "
                          "x = hi + lo); timed alone after an L2 flush"}

    # side measurement (not part of the step): each call alone, launched back
    # to back, its inputs rotated over enough device copies that every launch
    # reads them from HBM (ceil(4 x L2 / working set) copies, none for the
    # latency-bound small GEMM): the per-call time without an event between
    # launches
    steady = None
    if not args.no_steady:
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        steady = {}
        for k in keys:
            p = probs[k]
            ws = works[k]["bytes"]
            copies = 1 if (k == "c1" or ws >= 4 * l2) else min(8, -(-4 * l2 // ws))
            sets = [p.device_inputs()] + [[t.clone() for t in p.device_inputs()] for _ in range(copies - 1)]
            n_iter = 50
            for i in range(3):
                p.call(sptr, sets[i % copies])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(n_iter):
                p.call(sptr, sets[i % copies])
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n_iter
            steady[k] = {"ms": ms, "frac_of_roofline": roof[k] * 1e3 / ms, "input_copies": int(copies)}
            del sets
        torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # per-call report and the dominant kernel's roofline
    calls = {}
    for k in keys:
        wk = works[k]
        secs = per_call[k] / 1e3
        entry = {"ms": per_call[k], "roofline_ms": roof[k] * 1e3,
                 "frac_of_roofline": roof[k] / secs if secs > 0 else None,
                 "achieved_gbs": wk["bytes"] / secs / 1e9 if secs > 0 else None,
                 "achieved_tflops": wk["flops"] / secs / 1e12 if secs > 0 else None,
                 "algorithmic_bytes": wk["bytes"], "algorithmic_flops": wk["flops"]}
        if "distinct_experts" in wk:
            entry["distinct_experts"] = wk["distinct_experts"]
        calls[k] = entry
    wk = works[dom]
    secs = per_call[dom] / 1e3
    if wk["bound"] in ("tensor",):
        achieved = wk["flops"] / secs / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": achieved / tensor_peak}
    else:
        achieved = wk["bytes"] / secs / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"]}
    roofline.update({"kernel": dom, "peak_source": peak_src,
                     "peak_kind": "burst" if roofline["bound"] == "tensor" else "copy",
                     "traffic": TRAFFIC.get(dom)})

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(workloads, roof_total, args.cpu_scale)

    # side measurements outside the step (bounded): the rows beyond the five
    # workloads, each with its roofline fraction and the clocks seen
    side = None
    if not args.no_sweeps and world == 1:
        side = {}
        torch.cuda.empty_cache()
        quick = argparse.Namespace(steps=5, warmup=2)
        t_side = time.perf_counter()
        for name, fn in (("skinny_gemv", sweep_skinny), ("route_crossover", sweep_crossover),
                         ("matmul_id_dtypes", sweep_dtypes), ("ffma_gemm", sweep_ffma),
                         ("c3_cublas_context", cublas_context)):
            side[name] = fn(quick, torch, gb, quick=True)
            torch.cuda.empty_cache()
        side["seconds"] = time.perf_counter() - t_side

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": statistics.median(step_ms) if step_ms else None,
        "ms_per_step_min": min(step_ms) if step_ms else None,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16/bf16 in, f32 accumulate (f32 for c1)",
        "data": "synthetic (seeded numpy, seed 0)",
        "config": step_config(keys, peaks),
        "roofline_ms_per_step": roof_total * 1e3, "launches_per_step": n_launch,
        "step_times_ms": step_ms,
        "step_times_timing": ("one event per timed step just before the dominant call: consecutive events are "
                              "one step apart (no extra event in the step)"),
        "calls": calls,
        "calls_timing": (f"{dom}: events around its launches in every timed step; the other "
                         f"calls: an instrumented pass of {split_steps} steps with an event "
                         "between every two launches (those events are kept out of the timed "
                         "steps)"),
        "calls_split_ms": per_call_split,
        "calls_steady": steady,
        "calls_steady_timing": ("each call alone, 50 launches back to back between two events, "
                                "inputs rotated over input_copies device copies so that every "
                                "launch reads them from HBM (not part of the step)"),
        "c5_single_rounding_option": single,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
        "clocks": clk, "wall_s_timed": wall,
        "side_sweeps": side,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# DRAM traffic per launch from ncu (dram__bytes_read.sum + dram__bytes_write.sum,
# bytes), by workload, for the kernel as it stands; absent until captured again
# after a change to that kernel.  c5: grouped_tc_kernel<1, 0> (tail units,
# double-buffered epilogue, four activation stages, evict-first row stores,
# programmatic launch behind the map), 2.0494 GB read + 0.2013 GB written, one
# capture of the default-precision launch.
TRAFFIC: dict = {"c5": 2_250_667_776}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, as it stands, on the machine's host cores
# ---------------------------------------------------------------------------

def step_config(keys, peaks) -> dict:
    """The workload description both arms print (static: no measured values)."""
    return {"workload": "hot path: " + " + ".join(NAMES[k] for k in keys),
            "calls_per_step": len(keys),
            "l2": "inputs larger than L2 between calls: c5 streams 1.88 GB, each call's inputs "
                  "evicted by the calls before it",
            "parallelism": "replicas (one process per GPU, no exchange step)",
            "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in peaks}}


def run_reference(args) -> None:
    """The oracle as it stands on the host cores.  Each step is one bounded
    sample of the step's workload: every output of c1, c2 and c4, a sample of
    the outputs of c3 and c5; `ms_per_step` is the time those steps took,
    `value` the metric with the two sampled calls extrapolated to all their
    outputs."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import oracle
    oracle.build()
    keys = [k for k in ORDER if k in args.only]
    peaks, _ = load_peaks()
    tensor_peak = peaks["bf16_tflops"]
    workloads = {k: synth.workload(NAMES[k]) for k in keys}
    roof_total = sum(roofline_seconds(work_of(k, workloads[k]), peaks, tensor_peak) for k in keys)
    scale = args.cpu_scale
    for _ in range(args.warmup):
        cpu_step(workloads, keys, REF_SAMPLE, scale)
    steps = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        steps.append(cpu_step(workloads, keys, REF_SAMPLE, scale))
    wall = time.perf_counter() - t0
    est = statistics.mean(st["est_step_seconds"] for st in steps)
    value = 100.0 * roof_total / est
    last = steps[-1]
    cpu = {"value": value, "unit": UNIT, "cores": last["cores"], "cpu_model": last["cpu_model"],
           "kind": "oracle", "sample": last["sample"] + " per step",
           "measured_seconds_per_step": wall / max(1, args.steps),
           "est_full_step_seconds": est, "calls": last["calls"]}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate (oracle)",
            "data": "synthetic (seeded numpy, seed 0)", "impl": "reference",
            "config": step_config(keys, peaks),
            "timing": ("ms_per_step: wall time of each timed step, one bounded sample of the workload (every "
                       "output of the small calls, sampled outputs of the large ones); value: the metric for "
                       f"the full step, the sampled calls extrapolated by output count ({est:.1f} s per full "
                       "step)"),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s_timed": wall}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# side sweeps: the rows beyond the five workloads (each call timed alone)
# ---------------------------------------------------------------------------

def _time_alone(call, torch, flush, steps, warmup):
    """Mean of max(steps, 12) calls, each timed with CUDA events after an L2
    flush.  A device-side spin (about 0.2 ms) is queued between the flush and
    the start event so that the host has enqueued the call before the GPU
    reaches the event: the interval holds the call's device time, not the
    host's argument marshalling and launch latency.  The mean, not the median:
    on this GPU one event interval reads in steps of about 2.05 us, and the
    mean of many readings resolves what a median of them rounds away."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(steps, 12)):
        flush.fill_(1)
        torch.cuda._sleep(400_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.mean(ts)


def _with_clocks(fn):
    """Run fn() with the SM clocks sampled; returns (result, clocks)."""
    import torch
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    try:
        res = fn()
    finally:
        clk = clocks.stop()
    return res, clk


def sweep_crossover(args, torch, gb, quick=False) -> dict:
    """Both expert-ID routes on the grouped workload's expert stack (128
    experts of bf16 [1536, 4096], top-8 Zipf(1.1) ids, SharedPerToken f32 x)
    over m tokens, each call timed alone after an L2 flush (median of
    args.steps calls), with the first m at which GroupedPrefill is faster, for
    callers that choose the route."""
    peaks, _ = load_peaks()
    E, top_k, k, n = 128, 8, 4096, 1536
    stride = n * k * 2
    g = torch.Generator(device="cuda").manual_seed(0)
    w = (torch.randn(E * n * k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ms = (1, 8, 32, 64, 512) if quick else (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)

    def run():
        rows = []
        for m in ms:
            ids_h = synth.distinct_ids(m, top_k, E, seed=m, zipf_s=1.1)
            ids = torch.from_numpy(ids_h.view(np.int32).reshape(-1).copy()).cuda()
            x = torch.randn(m * k, device="cuda", generator=g)
            out = torch.empty(m * top_k * n, device="cuda")
            distinct = int(len(np.unique(ids_h)))
            bytes_ = distinct * stride + x.numel() * 4 + ids.numel() * 4 + out.numel() * 4
            flops = 2 * m * top_k * n * k
            roof_us = max(bytes_ / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
            entry = {"m": m, "distinct_experts": distinct, "roofline_us": roof_us}
            for route, name in ((gb.ROUTE_DIRECT, "direct"), (gb.ROUTE_GROUPED_PREFILL, "grouped")):
                p = gb.make_params(m, n, k, top_k, E, stride, 0, 0, route)
                st, cap = gb.gbmm_matmul_id_capability("bf16", p)
                gb.check(st)
                sc = None
                if route == gb.ROUTE_GROUPED_PREFILL:
                    cnt = torch.empty(cap.expert_counts_bytes, dtype=torch.uint8, device="cuda")
                    rr = torch.empty(cap.routed_rows_bytes, dtype=torch.uint8, device="cuda")
                    sc = gb.make_scratch(cnt, cap.expert_counts_bytes, rr, cap.routed_rows_bytes, E, m)

                def call():
                    gb.check(gb.gbmm_matmul_id(p, "bf16", w, w.numel() * 2, x, x.numel() * 4, ids,
                                               ids.numel() * 4, out, out.numel() * 4, sc)[0])
                us = _time_alone(call, torch, flush, args.steps, args.warmup)
                entry[name + "_us"] = us
                entry[name + "_frac_of_roofline"] = roof_us / us
                entry[name + "_kernel"] = gb.gbmm_test_last_kernel()
            rows.append(entry)
        return rows

    rows, clk = _with_clocks(run)
    cross = next((r["m"] for r in rows if r["grouped_us"] < r["direct_us"]), None)
    return {"sweep": "matmul_id route crossover", "experts": E, "top_k": top_k, "k": k, "n": n,
            "weights": "bf16", "ids": "top-8 distinct Zipf(1.1)",
            "timing": "each call alone after an L2 flush, median of %d" % args.steps,
            "roofline": "max(bytes of the distinct experts read + x + ids + out / HBM peak, flops / burst "
                        "bf16 peak)", "rows": rows, "grouped_faster_from_m": cross, "clocks": clk}


def sweep_ffma(args, torch, gb, quick=False) -> dict:
    """The f32 GEMM on the FFMA pipe at compute-bound sizes (f32 has no
    tensor-core route here), each call timed alone after an L2 flush, with its
    fraction of the FFMA peak (152 SMs x 128 lanes x 2 flops at the sampled SM
    clock)."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)
    shapes = [(4096, 4096, 4096, 0, 0), (4096, 4096, 4096, 0, 1)]
    if not quick:
        shapes += [(4096, 4096, 4096, 1, 0), (4096, 4096, 4096, 1, 1), (2048, 2048, 2048, 0, 1)]

    def run():
        rows = []
        for (m, n, k, ta, tb) in shapes:
            a = torch.randn(m * k, device="cuda", generator=g) / np.sqrt(k)
            b = torch.randn(n * k, device="cuda", generator=g)
            c = torch.empty(m * n, device="cuda")
            lda, ldb = (m if ta else k), (k if tb else n)

            def call():
                gb.check(gb.gbmm_gemm("f32", 1, m, n, k, ta, tb, a, 0, lda, m * k, b, 0, ldb, n * k, c, 0, n,
                                      m * n))
            us = _time_alone(call, torch, flush, args.steps, args.warmup)
            rows.append({"m": m, "n": n, "k": k, "ta": ta, "tb": tb, "us": us,
                         "tflops": 2 * m * n * k / (us * 1e-6) / 1e12, "kernel": gb.gbmm_test_last_kernel()})
            del a, b, c
        return rows

    rows, clk = _with_clocks(run)
    peak = ffma_peak_tflops((clk or {}).get("sm_mhz") or 2070.0)
    for r in rows:
        r["ffma_peak_tflops"] = peak
        r["frac_of_ffma_peak"] = r["tflops"] / peak
    return {"sweep": "f32 GEMM on the FFMA pipe", "timing": "each call alone after an L2 flush, median of "
            "%d" % args.steps, "rows": rows, "clocks": clk}


def sweep_skinny(args, torch, gb, quick=False) -> dict:
    """The decode GEMV y[m, n] = x[m, k] W[n, k]^T (B stored [n, k], batch 1)
    for m = 1 .. 15 tokens on the decode workload's shape (n 11008, k 4096),
    f16 and bf16 (and f32 at m = 1), plus the other GEMV orientations of the
    same f16 matrix: each call timed alone after an L2 flush, with the kernel
    that served it and its fraction of the HBM roofline (bytes of W, x and
    y)."""
    peaks, _ = load_peaks()
    n, k = 11008, 4096
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)
    sets = ((("f16", torch.float16, (1, 2, 4, 8, 15)), ("bf16", torch.bfloat16, (1, 8)),
             ("f32", torch.float32, (1,))) if quick else
            (("f16", torch.float16, (1, 2, 3, 4, 6, 8, 12, 15)), ("bf16", torch.bfloat16, (1, 2, 4, 8, 15)),
             ("f32", torch.float32, (1,))))

    def run():
        rows = []
        for dt, tdt, ms in sets:
            size = synth.ITEMSIZE[dt]
            w = (torch.randn(n * k, device="cuda", generator=g) * 0.02).to(tdt)
            for m in ms:
                x = torch.randn(m * k, device="cuda", generator=g).to(tdt)
                y = torch.empty(m * n, device="cuda", dtype=tdt)

                def call():
                    gb.check(gb.gbmm_gemm(dt, 1, m, n, k, 0, 1, x, 0, k, m * k, w, 0, k, n * k, y, 0, n, m * n))
                us = _time_alone(call, torch, flush, args.steps, args.warmup)
                bytes_ = (n * k + m * k + m * n) * size
                rows.append({"dtype": dt, "m": m, "us": us, "gbs": bytes_ / (us * 1e-6) / 1e9,
                             "frac_of_hbm": bytes_ / (peaks["hbm_gbs"] * 1e9) / (us * 1e-6),
                             "kernel": gb.gbmm_test_last_kernel()})
        # the vector times B stored [k, n] (outputs contiguous in the matrix
        # rows), and n == 1 with A stored [m, k] or [k, m]
        w = (torch.randn(n * k, device="cuda", generator=g) * 0.02).half()
        x = torch.randn(k, device="cuda", generator=g).half()
        y = torch.empty(n, device="cuda", dtype=torch.float16)
        for label, args_ in (("m1_B_stored_kn", (1, n, k, 0, 0, x, k, k, w, n, n * k, y, n, n)),
                             ("n1_A_stored_mk", (n, 1, k, 0, 1, w, k, n * k, x, k, k, y, 1, n)),
                             ("n1_A_stored_km", (n, 1, k, 1, 1, w, n, n * k, x, k, k, y, 1, n))):
            mm, nn, kk, ta, tb, a_, lda, sa, b_, ldb, sb, c_, ldc, sc = args_

            def call():
                gb.check(gb.gbmm_gemv("f16", 1, mm, nn, kk, ta, tb, a_, 0, lda, sa, b_, 0, ldb, sb, c_, 0, ldc,
                                      sc))
            us = _time_alone(call, torch, flush, args.steps, args.warmup)
            bytes_ = (n * k + k + n) * 2
            rows.append({"dtype": "f16", "orientation": label, "us": us, "gbs": bytes_ / (us * 1e-6) / 1e9,
                         "frac_of_hbm": bytes_ / (peaks["hbm_gbs"] * 1e9) / (us * 1e-6),
                         "kernel": gb.gbmm_test_last_kernel()})
        return rows

    rows, clk = _with_clocks(run)
    return {"sweep": "skinny decode GEMV", "n": n, "k": k, "layout": "B stored [n, k], batch 1 (plus the rows "
            "with an orientation)", "timing": "each call alone after an L2 flush, median of %d" % args.steps,
            "rows": rows, "clocks": clk}


def sweep_dtypes(args, torch, gb, quick=False) -> dict:
    """The expert-ID matmul for every weight dtype, input layout and id
    multiplicity the capability accepts: Direct on a decode shape (4 tokens x
    top-8 of 64 experts, k 2048, n 1408) and GroupedPrefill on a prefill shape
    (512 tokens, same experts), each call timed alone after an L2 flush, with
    its fraction of the roofline (HBM bytes of the experts the call reads, x,
    ids and out; tensor flops at the burst bf16 peak for 16-bit weights, the
    FFMA peak for f32 weights)."""
    peaks, _ = load_peaks()
    tensor_peak = peaks["bf16_tflops"]
    E, top_k, k, n = 64, 8, 2048, 1408
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)

    def run():
        rows = []
        for wdt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16), ("f32", torch.float32)):
            size = synth.ITEMSIZE[wdt]
            w = (torch.randn(E * n * k, device="cuda", generator=g) * 0.02).to(tdt)
            cases = [("direct", 4, 0, 0), ("direct", 4, 1, 0), ("direct", 4, 0, 1),
                     ("grouped", 512, 0, 0), ("grouped", 512, 1, 0)]
            for route_name, m, layout, mult in cases:
                route = gb.ROUTE_DIRECT if route_name == "direct" else gb.ROUTE_GROUPED_PREFILL
                ids_h = (synth.repeat_ids(m, top_k, E, seed=m) if mult else synth.distinct_ids(m, top_k, E, seed=m))
                ids = torch.from_numpy(ids_h.view(np.int32).reshape(-1).copy()).cuda()
                x_rows = m if layout == 0 else m * top_k
                x = torch.randn(x_rows * k, device="cuda", generator=g)
                out = torch.empty(m * top_k * n, device="cuda")
                p = gb.make_params(m, n, k, top_k, E, n * k * size, layout, mult, route)
                st, cap = gb.gbmm_matmul_id_capability(wdt, p)
                gb.check(st)
                sc = None
                if route == gb.ROUTE_GROUPED_PREFILL:
                    cnt = torch.empty(cap.expert_counts_bytes, dtype=torch.uint8, device="cuda")
                    rr = torch.empty(cap.routed_rows_bytes, dtype=torch.uint8, device="cuda")
                    sc = gb.make_scratch(cnt, cap.expert_counts_bytes, rr, cap.routed_rows_bytes, E, m)

                def call():
                    gb.check(gb.gbmm_matmul_id(p, wdt, w, w.numel() * size, x, x.numel() * 4, ids,
                                               ids.numel() * 4, out, out.numel() * 4, sc)[0])
                us = _time_alone(call, torch, flush, args.steps, args.warmup)
                distinct = int(len(np.unique(ids_h)))
                bytes_ = distinct * n * k * size + x.numel() * 4 + ids.numel() * 4 + out.numel() * 4
                flops = 2 * m * top_k * n * k
                peak_tf = ffma_peak_tflops() if wdt == "f32" else tensor_peak
                roof = max(bytes_ / (peaks["hbm_gbs"] * 1e9), flops / (peak_tf * 1e12))
                rows.append({"weights": wdt, "route": route_name, "m": m,
                             "layout": "Slotted" if layout else "SharedPerToken",
                             "ids": "MayRepeat" if mult else "DistinctPerToken", "distinct_experts": distinct,
                             "us": us, "roofline_us": roof * 1e6, "frac_of_roofline": roof / (us * 1e-6),
                             "kernel": gb.gbmm_test_last_kernel()})
            del w
        return rows

    rows, clk = _with_clocks(run)
    return {"sweep": "matmul_id weight dtypes, layouts and multiplicity", "experts": E, "top_k": top_k,
            "k": k, "n": n, "timing": "each call alone after an L2 flush, median of %d" % args.steps,
            "rows": rows, "clocks": clk}


def cublas_context(args, torch, gb, quick=False) -> dict:
    """Context only (never a baseline of ours): cuBLAS through torch.bmm on
    the batched f16 GEMM workload's shape (4 x 4096^3, B stored [n, k]), timed
    alone after an L2 flush and back to back, beside this library's call of
    the same shape timed the same way."""
    b, m, n, k = 4, 4096, 4096, 4096
    g = torch.Generator(device="cuda").manual_seed(0)
    a = (torch.randn(b * m * k, device="cuda", generator=g) / 64).half()
    bt = (torch.randn(b * n * k, device="cuda", generator=g) / 64).half()
    c = torch.empty(b * m * n, device="cuda", dtype=torch.float16)
    a3, b3 = a.view(b, m, k), bt.view(b, n, k)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def ours():
        gb.check(gb.gbmm_gemm("f16", b, m, n, k, 0, 1, a, 0, k, m * k, bt, 0, k, n * k, c, 0, n, m * n))

    def theirs():
        torch.bmm(a3, b3.transpose(1, 2))

    flops = 2 * b * m * n * k
    out = {"shape": "f16 batch 4, 4096^3, B stored [n, k]", "note": "cuBLAS (torch.bmm) as context only"}
    for name, fn in (("gbmm", ours), ("cublas", theirs)):
        us = _time_alone(fn, torch, flush, args.steps, args.warmup)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            fn()
        e1.record()
        torch.cuda.synchronize()
        b2b = e0.elapsed_time(e1) * 1e3 / 20
        out[name] = {"us_alone": us, "us_back_to_back": b2b, "tflops_alone": flops / (us * 1e-6) / 1e12,
                     "tflops_back_to_back": flops / (b2b * 1e-6) / 1e12}
    return out


def run_sweep(args, fn) -> None:
    import torch
    from gemv_moe_expert_gb300 import binding as gb
    from gemv_moe_expert_gb300 import build
    build.build()
    gb.load()
    print(json.dumps(fn(args, torch, gb, quick=False)), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", default=",".join(ORDER))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-scale", type=float, default=1.0)
    ap.add_argument("--no-options", action="store_true", help="skip the opt-in mode side timings")
    ap.add_argument("--no-steady", action="store_true", help="skip the per-call back-to-back timings")
    ap.add_argument("--no-sweeps", action="store_true",
                    help="skip the side sweeps (skinny GEMV, route crossover, matmul_id dtypes, FFMA GEMM)")
    ap.add_argument("--sweep", choices=["crossover", "skinny", "dtypes", "ffma"], default=None,
                    help="instead of the step: crossover = Direct against GroupedPrefill for m = 1..512; "
                         "skinny = the decode GEMV for m = 1..15; dtypes = the expert-ID matmul for every "
                         "weight dtype, input layout and id multiplicity; ffma = the f32 GEMM at 4096^3")
    args = ap.parse_args()
    args.only = [k.strip() for k in args.only.split(",") if k.strip()]
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.sweep is not None:
        run_sweep(args, {"crossover": sweep_crossover, "skinny": sweep_skinny, "dtypes": sweep_dtypes,
                         "ffma": sweep_ffma}[args.sweep])
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
