#!/usr/bin/env python3
"""Throughput benchmark of the sliced tensor-parallel MLP layer on GB300.

One step = one domino_mlp_fwd over one batch of the workload (GEMM1 + GEMM2 +
shard-sum for every chunk and slice), inputs resident in HBM.  Prints ONE JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--mu MU]
                  [--schedule fused|streams|serial] [--plan] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one independent replica per GPU (the
workload has no exchange between GPUs: weak scaling, no data-path collective;
the only collectives are the timing barrier and the max over ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The device-code sources each kernel kind is built from: a stored ncu capture of a kernel applies while the
# hash of its own sources is unchanged.
_GEMM_SOURCES = ("common.h", "epilogue.cuh", "gemm.cu", "gemm.h", "gemm_pair.cu", "ptx.cuh")
KERNEL_SOURCES = {
    "fused": ("common.h", "epilogue.cuh", "fused.cu", "gemm.h", "ptx.cuh"),
    "bwd_dx_fused": ("common.h", "epilogue.cuh", "fused.cu", "gemm.h", "ptx.cuh"),
    "gemm1": _GEMM_SOURCES, "gemm2": _GEMM_SOURCES,
    "bwd_dh": _GEMM_SOURCES, "bwd_dx": _GEMM_SOURCES, "bwd_dw": _GEMM_SOURCES,
    "shard_sum": ("common.h", "gemm.h", "ptx.cuh", "shard_sum.cu"),
    "attn": ("attn.cu", "attn.h", "common.h", "ptx.cuh"),
}


def kernel_source_hash(kernel_kind):
    """Hash of the device-code sources of one kernel kind, to tell whether a stored ncu capture still applies."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "communication_overlap_domino_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel_kind]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_kind, workload, mu):
    """DRAM bytes per launch from a committed ncu capture, if it was taken at the same number of chunks (a launch
    covers one chunk, or all of them) and matches the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("kernels", {}).get(f"{workload}/{kernel_kind}")
    if entry is None or kernel_kind not in KERNEL_SOURCES or entry.get("mu") != mu:
        return None
    if entry.get("source_hash") != kernel_source_hash(kernel_kind):
        return None
    return entry.get("dram_bytes_per_launch")


def device_info(dev):
    """The GPU the line was measured on: the L2 size and the SM count bear on how the kernels' DRAM re-reads and
    grids come out, which differ between boxes."""
    import torch

    pr = torch.cuda.get_device_properties(dev)
    return {"name": pr.name, "sms": pr.multi_processor_count, "l2_bytes": int(getattr(pr, "L2_cache_size", 0)),
            "memory_bytes": int(pr.total_memory)}


def tensor_peak_for(peaks, launch_s):
    """The bf16 denominator for a kernel whose launches last launch_s seconds: the burst figure (a GEMM
    timed alone, best of 10) for launches under a second, the sustained one (seconds back to back under
    the power cap) for longer ones.  Returns (peak, which)."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    return (burst, "bf16_tflops") if launch_s < 1.0 else (sustained, "bf16_tflops_sustained")


# ------------------------------------------------------------------- NVTX

# The timed region is an NVTX push/pop range of this name, so that a profiler's launch list can be limited
# to it (ncu --nvtx --nvtx-include "timed_region/").
TIMED_RANGE = "timed_region"


def nvtx_push(name):
    try:
        import torch
        torch.cuda.nvtx.range_push(name)
    except Exception:  # NVTX is optional: the timing does not depend on it
        pass


def nvtx_pop():
    try:
        import torch
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.mark = 0
        self.in_timed = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def ready(self, work, timeout_s=5.0):
        """Runs `work` (one untimed step of the same load, synchronised) until nvidia-smi has
        delivered its first sample, then marks where the timed region's samples begin."""
        import torch
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            work()
            torch.cuda.synchronize()
        self.mark = len(self.lines)

    def top_up(self, work, n=3, timeout_s=5.0):
        """Ends the timed region's samples.  A region too short for n samples at the 100 ms
        period is followed by untimed steps of the same load until n samples have arrived."""
        import torch
        self.in_timed = len(self.lines) - self.mark
        t0 = time.perf_counter()
        while self.proc is not None and len(self.lines) - self.mark < n and time.perf_counter() - t0 < timeout_s:
            work()
            torch.cuda.synchronize()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines[self.mark:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
               "samples": len(sm)}
        if self.in_timed is not None and self.in_timed < len(sm):
            out["samples_in_timed_region"] = self.in_timed
            out["note"] = "timed region shorter than the samples asked for: the rest come from untimed steps " \
                          "of the same load right after it"
        return out


# ------------------------------------------------------ tensor-core probe

def tensor_probe(clk, repeats=3, mmas=1 << 17):
    """Best of `repeats` runs of domino_tensor_peak (paired tcgen05 MMAs alone, every co-resident
    2-CTA cluster), with the per-SM rate per clock it measures and the theoretical rate
    SMs x that rate x SM clock, at the clock sampled under the timed region's load and at the
    maximum SM clock."""
    from communication_overlap_domino_gb300 import binding as b
    runs = [b.tensor_peak(mmas) for _ in range(repeats)]
    best = max(runs, key=lambda r: r["tflops"])
    fpc = max(r["flops_per_clk_sm"] for r in runs)
    out = {"tflops": round(best["tflops"], 1), "sm_mhz_in_probe": round(best["sm_mhz"], 1),
           "flops_per_clk_per_sm": round(fpc, 1), "clusters": best["clusters"], "num_sms": best["num_sms"],
           "mmas_per_cluster": mmas, "mma": "tcgen05.mma cta_group::2 kind::f16 256x256x16, bf16 -> fp32"}
    if clk:
        out["theoretical_tflops_at_load_clock"] = round(best["num_sms"] * fpc * clk["sm_mhz"] * 1e6 / 1e12, 1)
        out["theoretical_tflops_at_max_clock"] = round(best["num_sms"] * fpc * clk["sm_max_mhz"] * 1e6 / 1e12, 1)
    return out


# ------------------------------------------------------------ CPU baseline

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model():
    """The host CPU's name (x86 'model name', or the Arm implementer/part ids) and its logical core count."""
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
        if m:
            name = m.group(1).strip()
        else:
            imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
            part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
            if imp and part:
                name = f"{os.uname().machine} implementer {imp.group(1)} part {part.group(1)}"
    except OSError:
        pass
    return {"model": name or os.uname().machine, "logical_cores": os.cpu_count()}


def oracle_step(w, f64, X, dY):
    """One oracle step on a row sample: forward, plus backward for training workloads."""
    import oracle
    A = (f64["Wg"], f64["Wu"]) if w.act == "swiglu" else f64["A"]
    if w.bwd:
        return oracle.mlp_bwd(X, A, f64["B"], dY, w.act)
    return oracle.mlp_fwd(X, A, f64["B"], w.act)


def oracle_row_sample(w, t, target_s):
    """Times the fp64 oracle on a row sample sized for about target_s.

    Rows are independent in the block (and the weight gradients are sums over
    rows), so the sample's flops scale exactly with its row count.
    Returns (rows, seconds, flops)."""
    f64 = {k: v.to("cpu").double().numpy() for k, v in t.items() if k not in ("X", "dY")}
    rows = min(w.M, 32)
    step_flops = w.fwd_flops() + (w.bwd_flops() if w.bwd else 0)
    while True:
        X = t["X"][:rows].double().numpy()
        dY = t["dY"][:rows].double().numpy() if w.bwd else None
        t0 = time.perf_counter()
        oracle_step(w, f64, X, dY)
        dt = time.perf_counter() - t0
        flops = step_flops * rows / w.M
        if dt >= 0.5 * target_s or rows >= w.M:
            return rows, dt, flops
        rows = int(min(w.M, max(rows * 2, rows * target_s / max(dt, 1e-3))))


# -------------------------------------------------------------- multi-rank

def max_over_ranks(value_ms, world, device=None):
    """The slowest rank's time: every rank runs its own replica of the workload
    (weak scaling), so the job's step time is the maximum over ranks."""
    if world <= 1:
        return float(value_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, max_ms):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- our arm

def timeline_stats(records):
    """Per call: span of all launches, GEMM-busy time, exposed (non-GEMM) time."""
    calls = {}
    for r in records:
        calls.setdefault(r["call"], []).append(r)
    spans, exposed = [], []
    for recs in calls.values():
        lo = min(r["start_ms"] for r in recs)
        hi = max(r["end_ms"] for r in recs)
        ivs = sorted((r["start_ms"], r["end_ms"]) for r in recs if r["kind"] != "shard_sum")
        busy, cur_s, cur_e = 0.0, None, None
        for s, e in ivs:
            if cur_e is None or s > cur_e:
                if cur_e is not None:
                    busy += cur_e - cur_s
                cur_s, cur_e = s, e
            else:
                cur_e = max(cur_e, e)
        if cur_e is not None:
            busy += cur_e - cur_s
        spans.append(hi - lo)
        exposed.append(max(0.0, (hi - lo) - busy))
    return statistics.mean(spans), statistics.mean(exposed)


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from communication_overlap_domino_gb300 import binding as b
    from communication_overlap_domino_gb300 import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    t = wl.generate(w, seed=0)
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    del A
    X = t["X"].to(dev)
    Y = torch.empty((w.M, w.d), dtype=torch.bfloat16, device=dev)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, args.schedule)
    ws = torch.zeros(b.workspace_size(desc, with_bwd=w.bwd), dtype=torch.uint8, device=dev)
    if w.bwd:  # training step: forward keeping the pre-activations, then backward
        dY = t["dY"].to(dev)
        saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=dev)
        dX = torch.empty_like(X)
        dA_sh = [torch.empty_like(a) for a in A_sh]
        dB_sh = [torch.empty_like(x) for x in B_sh]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(timed=False, x=X, dy=None, y=None, dx=None):
        b.mlp_fwd(x, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                  schedule=args.schedule, Y=Y if y is None else y, workspace=ws, kernel_times=timed,
                  saved=saved if w.bwd else None)
        if w.bwd:
            b.mlp_bwd(x, A_sh, B_sh, dY if dy is None else dy, saved, F=w.F, mu=w.mu, act=w.act,
                      partial=w.partial, out_slices=w.slices, schedule=args.schedule, dX=dX if dx is None else dx,
                      dA_shards=dA_sh, dB_shards=dB_sh, workspace=ws, kernel_times=timed)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier(device_ids=[local_rank])

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    st = b.query_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {b.STATUS.get(st)}")

    # ---- timed region: K steps, L2 flushed between steps (outside the step events)
    b.kernel_times_reset()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[local_rank]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local_rank
    clocks = ClockSampler(gpu_index)
    clocks.start()
    load = lambda: (flush.zero_(), step())  # noqa: E731
    clocks.ready(load)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    wall0 = time.perf_counter()
    nvtx_push(TIMED_RANGE)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step(timed=True)
        ev[i][1].record(stream)
    barrier()
    nvtx_pop()
    wall = time.perf_counter() - wall0
    clocks.top_up(load)
    clk = clocks.stop()
    probe = tensor_probe(clk)
    st = b.query_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {b.STATUS.get(st)}")
    step_ms = [s.elapsed_time(e) for s, e in ev]
    mean_ms = statistics.mean(step_ms)
    records = b.kernel_times()
    mean_ms = max_over_ranks(mean_ms, world, dev)

    # ---- fused schedule: reduction time left after the last GEMM tile, from the
    # kernel's own %globaltimer stamps (read back after each of a few extra calls)
    fused_exposed = None
    fused_exposed_parts = None
    if args.schedule == "fused":
        ex_f, ex_b = [], []
        for _ in range(20):
            b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, schedule="fused", Y=Y,
                      workspace=ws, saved=saved if w.bwd else None)
            tl = b.read_timeline(ws)
            ex_f.append(max(0, tl["reduce_end_ns"] - tl["gemm_end_ns"]) * 1e-6)
            if w.bwd:  # the backward's partial input gradients and their shard-sum: one cooperative launch
                b.mlp_bwd(X, A_sh, B_sh, dY, saved, F=w.F, mu=w.mu, act=w.act, partial=w.partial,
                          out_slices=w.slices, schedule="fused", dX=dX, dA_shards=dA_sh, dB_shards=dB_sh,
                          workspace=ws)
                tl = b.read_timeline(ws)
                ex_b.append(max(0, tl["reduce_end_ns"] - tl["gemm_end_ns"]) * 1e-6)
        fused_exposed = statistics.mean(ex_f) + (statistics.mean(ex_b) if ex_b else 0.0)
        fused_exposed_parts = {"fwd_us": round(1e3 * statistics.mean(ex_f), 2)}
        if ex_b:
            fused_exposed_parts["bwd_us"] = round(1e3 * statistics.mean(ex_b), 2)

    # ---- A/B measure of the reduction's cost: the same call without the shard-sum, alternating with the full
    # call (L2 flushed before each).  domino_mlp_fwd_partials runs the same GEMM tiles in the same order and
    # writes the same partials, which are its result; the difference in mean duration is what the shard-sum
    # adds to the layer, including its slowing of the GEMM tiles it runs beside.
    ab = None
    if not w.bwd and args.ab_pairs > 0:
        zdt = torch.float32 if w.partial == "f32" else torch.bfloat16
        Zab = [torch.empty((w.M, w.d), dtype=zdt, device=dev) for _ in range(w.P)]
        kw_ab = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule=args.schedule,
                     workspace=ws)
        ev_ab = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.ab_pairs)] for _ in range(2)]
        for i in range(args.ab_pairs):
            for which in (0, 1):
                flush.zero_()
                ev_ab[which][i][0].record(stream)
                if which == 0:
                    b.mlp_fwd(X, A_sh, B_sh, Y=Y, **kw_ab)
                else:
                    b.mlp_fwd_partials(X, A_sh, B_sh, Z_shards=Zab, **kw_ab)
                ev_ab[which][i][1].record(stream)
        torch.cuda.synchronize()
        full_ms = statistics.mean(a.elapsed_time(e) for a, e in ev_ab[0])
        part_ms = statistics.mean(a.elapsed_time(e) for a, e in ev_ab[1])
        ab = {"full_ms": round(full_ms, 4), "partials_ms": round(part_ms, 4), "pairs": args.ab_pairs,
              "exposed_us": round(1e3 * (full_ms - part_ms), 2),
              "method": "mean duration of domino_mlp_fwd minus that of domino_mlp_fwd_partials (same schedule, "
                        "same GEMM tiles, no shard-sum), calls alternating, L2 flushed before each"}
        del Zab
        if b.query_device_status(ws) != 0:
            raise RuntimeError("device status after the A/B calls")

    # ---- the L2 flush alone, for reading the end-to-end numbers (which contain it)
    fl_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for s_, e_ in fl_ev:
        s_.record(stream)
        flush.zero_()
        e_.record(stream)
    torch.cuda.synchronize()
    flush_ms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in fl_ev)

    # ---- end to end: pinned host X in, Y out, copies inside the timed region
    e2e_steps = max(3, min(args.steps, 200))
    Xh = t["X"].pin_memory()
    Yh = torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory()
    Xd = torch.empty_like(X)
    if w.bwd:
        dYh = t["dY"].pin_memory()
        dXh = torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory()
        dYd = torch.empty_like(X)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.zero_()
        ev2[i][0].record(stream)
        Xd.copy_(Xh, non_blocking=True)
        if w.bwd:
            dYd.copy_(dYh, non_blocking=True)
            step(x=Xd, dy=dYd)
            dXh.copy_(dX, non_blocking=True)
        else:
            step(x=Xd)
        Yh.copy_(Y, non_blocking=True)
        ev2[i][1].record(stream)
    barrier()
    e2e_serial_ms = statistics.mean(s.elapsed_time(e) for s, e in ev2)
    e2e_serial_ms = max_over_ranks(e2e_serial_ms, world, dev)
    if not torch.equal(Yh, Y.cpu()):
        raise RuntimeError("end-to-end output differs from the device result")

    # ---- end to end, pipelined as a streaming caller runs it: every step still
    # uploads its own input and downloads its own result inside the timed region,
    # but on a copy stream, so step i+1's upload and step i's download overlap
    # the compute of the neighbouring steps (double-buffered device and host
    # buffers).  The L2 flush stays on the compute stream, inside the region.
    copy = torch.cuda.Stream(device=dev)       # uploads
    copy_back = torch.cuda.Stream(device=dev)  # downloads (the two directions run concurrently)
    Xb = [torch.empty_like(X) for _ in range(2)]
    Yb = [torch.empty_like(Y) for _ in range(2)]
    Yhb = [torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    if w.bwd:
        dYb = [torch.empty_like(X) for _ in range(2)]
        dXb = [torch.empty_like(X) for _ in range(2)]
        dXhb = [torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    up = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier()
    e_start.record(stream)
    copy.wait_event(e_start)
    copy_back.wait_event(e_start)

    downloaded = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        with torch.cuda.stream(copy):
            if i >= 2:  # buffer i % 2 was last read by step i - 2's compute
                copy.wait_event(done[i % 2])
            Xb[i % 2].copy_(Xh, non_blocking=True)
            if w.bwd:
                dYb[i % 2].copy_(dYh, non_blocking=True)
            up[i % 2].record(copy)

    upload(0)
    if e2e_steps > 1:
        upload(1)
    for i in range(e2e_steps):
        j = i % 2
        flush.zero_()
        stream.wait_event(up[j])
        if i >= 2:  # step i - 2's result buffer must have been downloaded
            stream.wait_event(downloaded[j])
        step(x=Xb[j], y=Yb[j], dy=dYb[j] if w.bwd else None, dx=dXb[j] if w.bwd else None)
        done[j].record(stream)
        with torch.cuda.stream(copy_back):
            copy_back.wait_event(done[j])
            Yhb[j].copy_(Yb[j], non_blocking=True)
            if w.bwd:
                dXhb[j].copy_(dXb[j], non_blocking=True)
            downloaded[j].record(copy_back)
        if i + 2 < e2e_steps:
            upload(i + 2)
    e_end.record(copy_back)
    stream.wait_event(e_end)
    barrier()
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    if not torch.equal(Yhb[(e2e_steps - 1) % 2], Y.cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the device result")

    if rank != 0:
        return None

    # ---- per-kernel durations from the live events of the timed region
    peaks, peak_src = load_peaks()
    nact = 2 if w.act == "swiglu" else 1
    ds_ = w.d // w.slices

    def launch_flops(r):  # algorithmic GEMM flops of one launch (all shards)
        return {"fused": float(w.fwd_flops()),
                "gemm1": 2.0 * w.Mc * w.d * w.F * nact, "gemm2": 2.0 * w.Mc * w.F * ds_,
                "bwd_dh": 2.0 * w.M * w.d * w.F, "bwd_dx": 2.0 * w.Mc * nact * w.F * ds_,
                "bwd_dx_fused": 2.0 * w.M * nact * w.F * w.d,
                "bwd_dw": 2.0 * w.M * w.d * w.F * (nact if r["slice"] == 0 else 1)}.get(r["kind"], 0.0)

    psize = 4 if w.partial == "f32" else 2
    ss_bytes = (w.P * psize + 2) * w.Mc * ds_
    kinds = {}
    for r in records:
        k = kinds.setdefault(r["kind"], {"launches": 0, "total_ms": 0.0, "flops": 0.0})
        k["launches"] += 1
        k["total_ms"] += r["end_ms"] - r["start_ms"]
        k["flops"] += launch_flops(r)
    for k in kinds.values():
        k["avg_us"] = 1e3 * k["total_ms"] / k["launches"]
    dominant = max((k for k in kinds if k != "shard_sum"), key=lambda k: kinds[k]["total_ms"])
    dom_tflops = kinds[dominant]["flops"] / (kinds[dominant]["total_ms"] * 1e-3) / 1e12
    dom_flops_per_launch = kinds[dominant]["flops"] / kinds[dominant]["launches"]
    peak_tf, peak_key = tensor_peak_for(peaks, kinds[dominant]["avg_us"] * 1e-6)
    sustained_tf = float(peaks.get("bf16_tflops_sustained", peak_tf))
    ss_gbs = ss_bytes / (kinds["shard_sum"]["avg_us"] * 1e-6) / 1e9 if "shard_sum" in kinds else None
    span_ms, exposed_ms = timeline_stats(records)
    calls_per_step = 2 if w.bwd else 1
    span_ms *= calls_per_step
    exposed_ms *= calls_per_step
    if fused_exposed is not None:  # the fused kernels reduce inside the launch: use their device timelines
        exposed_ms = fused_exposed

    flops = w.fwd_flops() + (w.bwd_flops() if w.bwd else 0)
    value = whole_job_tflops(flops, world, mean_ms)
    line = {
        "metric": "sliced TP-MLP layer TFLOP/s at 1 GB300 (% BF16 peak); exposed shard-reduce time/layer",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) activations, N(0,0.02) weights, bf16",
        "config": {"workload": w.name, "M": w.M, "d": w.d, "F": w.F, "P": w.P, "mu": w.mu, "act": w.act,
                   "partials": w.partial, "out_slices": w.slices, "schedule": args.schedule,
                   "l2": "flushed between steps (256 MiB write outside the step events)",
                   **({"plan": args.plan_result} if getattr(args, "plan_result", None) else {})},
        "pct_of_bf16_peak": round(100.0 * value / world / peak_tf, 2),
        "pct_of_bf16_sustained": round(100.0 * value / world / sustained_tf, 2),
        "exposed_reduce_us_per_layer": round(1e3 * exposed_ms, 2),
        "exposed_reduce_frac": round(exposed_ms / span_ms, 4) if span_ms > 0 else None,
        "exposed_reduce_method": "fused: the kernel's own %globaltimer stamps, last GEMM tile end to last "
                                 "shard-sum piece end; streams/serial: call span minus the union of GEMM launch "
                                 "intervals (CUDA events)",
        "exposed_reduce_us_per_call": fused_exposed_parts,
        "exposed_reduce_ab_us_per_layer": None if ab is None else ab["exposed_us"],
        "exposed_reduce_ab": ab,
        "roofline": {
            "kernel": {"fused": "fused_fwd_pair_kernel (both projections and the shard-sum, one launch)",
                       "bwd_dx_fused": "fused_fwd_pair_kernel, backward mode (partial input gradients of every "
                                       "chunk and their shard-sum, one launch)"}.get(
                dominant, f"gemm_pair_kernel ({dominant})"),
            "note": "achieved = algorithmic flops of the kernel's launches / their summed event durations; peak = "
                    "the burst bf16 figure for launches under a second, else the sustained one",
            "bound": "tensor",
            "achieved": round(dom_tflops, 2),
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": round(dom_tflops / peak_tf, 4),
            "peak_source": f"{peak_src} {peak_key}",
            "avg_launch_us": round(kinds[dominant]["avg_us"], 2),
            "frac_of_sustained": round(dom_tflops / sustained_tf, 4),
            "flops_per_launch": dom_flops_per_launch,
            "traffic": ncu_traffic(dominant, w.name, w.mu),
            "frac_of_mma_probe": round(dom_tflops / probe["tflops"], 4),
        },
        "tensor_probe": probe,
        "device": device_info(dev),
        "shard_sum": None if ss_gbs is None else {
            "bound": "hbm",
            "achieved": round(ss_gbs, 1),
            "peak": float(peaks.get("hbm_gbs")),
            "unit": "GB/s",
            "frac": round(ss_gbs / float(peaks.get("hbm_gbs")), 4),
            "bytes_per_launch": ss_bytes,
            "traffic": ncu_traffic("shard_sum", w.name, w.mu),
        },
        "kernels": {k: {"launches": v["launches"], "avg_us": round(v["avg_us"], 2),
                        "tflops": round(v["flops"] / (v["total_ms"] * 1e-3) / 1e12, 1) if v["flops"] else None,
                        "share": round(v["total_ms"] / sum(x["total_ms"] for x in kinds.values()), 4)}
                    for k, v in kinds.items()},
        "gpu_launches": len(records),
        "e2e": {"value": round(whole_job_tflops(flops, world, e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": w.M * w.d * 2 * calls_per_step,
                "d2h_bytes_per_step": w.M * w.d * 2 * calls_per_step,
                "ms_per_step": round(e2e_ms, 4),
                "l2_flush_ms_per_step": round(flush_ms, 4),
                "mode": "pipelined: each step uploads its input from pinned host memory and downloads its result "
                        "on two copy streams, overlapping the neighbouring steps' compute (double-buffered); "
                        "each step also contains the 256 MiB L2 flush"},
        "e2e_serial": {"value": round(whole_job_tflops(flops, world, e2e_serial_ms), 2), "unit": "TFLOP/s",
                       "ms_per_step": round(e2e_serial_ms, 4),
                       "mode": "upload, compute, download in order on one stream each step (L2 flush outside the events)"},
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        rows, dt, fl = oracle_row_sample(w, t, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(fl / dt / 1e12, 5), "unit": "TFLOP/s", "cores": blas_threads(),
                                "cpu": cpu_model(),
                                "kind": "oracle",
                                "sample": f"fp64 oracle {'forward+backward' if w.bwd else 'forward'} on {rows} "
                                          f"of {w.M} rows ({dt:.1f} s; rows are "
                                          f"independent, flops scale with rows)"}
    return line


# --------------------------------------------------------- attention block

def run_attn(args, w, rank, world, local_rank):
    """The sliced tensor-parallel attention block (domino_attn_fwd): projection,
    flash-style attention core, output projection, shard-sum, per chunk."""
    import torch

    from communication_overlap_domino_gb300 import binding as b
    from communication_overlap_domino_gb300 import workloads as wl
    import oracle.attention as att

    schedule = args.schedule
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    t = wl.generate_attn(w, seed=0)
    qkv_sh, o_sh = b.shard_attn_weights(t["Wqkv"].to(dev), t["Wo"].to(dev), w.H, w.P)
    X = t["X"].to(dev)
    Y = torch.empty((w.M, w.d), dtype=torch.bfloat16, device=dev)
    desc = b.make_attn_desc(w.B, w.S, w.d, w.H, w.P, w.mu, w.partial, schedule)
    ws = torch.zeros(b.attn_workspace_size(desc), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(timed=False, x=X, y=Y):
        b.attn_fwd(x, qkv_sh, o_sh, S=w.S, H=w.H, mu=w.mu, partial=w.partial, schedule=schedule, Y=y,
                   workspace=ws, kernel_times=timed)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if b.query_device_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    b.kernel_times_reset()
    clocks = ClockSampler(local_rank)
    clocks.start()
    load = lambda: (flush.zero_(), step())  # noqa: E731
    clocks.ready(load)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    nvtx_push(TIMED_RANGE)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step(timed=True)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    nvtx_pop()
    wall = time.perf_counter() - wall0
    clocks.top_up(load)
    clk = clocks.stop()
    probe = tensor_probe(clk)
    if b.query_device_status(ws) != 0:
        raise RuntimeError("device status after the timed region")
    mean_ms = max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in ev), world, dev)
    records = b.kernel_times()

    # FUSED: the last chunk's output projection and shard-sum are one cooperative launch whose timeline (3 words:
    # ~start, last GEMM tile end, last shard-sum end) sits at workspace byte 64 + 24 k; the earlier chunks'
    # shard-sums run beside the next chunk as in STREAMS (their exposure is in the launch timeline below)
    fused_tail = None
    if schedule == "fused":
        tails = []
        k = w.mu - 1
        for _ in range(20):
            step()
            torch.cuda.synchronize()
            r = ws[64 + 24 * k:64 + 24 * k + 24].clone().view(torch.int64).cpu()
            tails.append(max(0, int(r[2]) - int(r[1])) * 1e-6)
        fused_tail = statistics.mean(tails)
    Xh = t["X"].pin_memory()
    Yh = torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory()
    Xd = torch.empty_like(X)
    e2e_steps = max(3, min(args.steps, 50))
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.zero_()
        ev2[i][0].record(stream)
        Xd.copy_(Xh, non_blocking=True)
        step(x=Xd)
        Yh.copy_(Y, non_blocking=True)
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in ev2), world, dev)
    if not torch.equal(Yh, Y.cpu()):
        raise RuntimeError("end-to-end output differs from the device result")

    # ---- end to end, pipelined as a streaming caller runs it (as for the MLP): every step uploads its own input
    # and downloads its own result inside the timed region, on copy streams, double-buffered, so the copies of
    # neighbouring steps overlap the compute; the L2 flush stays on the compute stream
    copy = torch.cuda.Stream(device=dev)
    copy_back = torch.cuda.Stream(device=dev)
    Xb = [torch.empty_like(X) for _ in range(2)]
    Yb = [torch.empty_like(Y) for _ in range(2)]
    Yhb = [torch.empty((w.M, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    up = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e_start.record(stream)
    copy.wait_event(e_start)
    copy_back.wait_event(e_start)

    def upload(i):
        with torch.cuda.stream(copy):
            if i >= 2:  # buffer i % 2 was last read by step i - 2's compute
                copy.wait_event(done[i % 2])
            Xb[i % 2].copy_(Xh, non_blocking=True)
            up[i % 2].record(copy)

    upload(0)
    upload(1)
    for i in range(e2e_steps):
        j = i % 2
        flush.zero_()
        stream.wait_event(up[j])
        if i >= 2:  # step i - 2's result buffer must have been downloaded
            stream.wait_event(downloaded[j])
        step(x=Xb[j], y=Yb[j])
        done[j].record(stream)
        with torch.cuda.stream(copy_back):
            copy_back.wait_event(done[j])
            Yhb[j].copy_(Yb[j], non_blocking=True)
            downloaded[j].record(copy_back)
        if i + 2 < e2e_steps:
            upload(i + 2)
    e_end.record(copy_back)
    stream.wait_event(e_end)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / e2e_steps, world, dev)
    if not torch.equal(Yhb[(e2e_steps - 1) % 2], Y.cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the device result")
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    Mc = w.M // w.mu
    core_flops_chunk = 2 * 2 * (w.B // w.mu) * w.H * w.dh * (w.S * (w.S + 1) // 2)
    launch_flops = {"gemm1": 2.0 * Mc * w.d * 3 * w.H * w.dh, "attn": float(core_flops_chunk),
                    "gemm2": 2.0 * Mc * w.H * w.dh * w.d, "attn_out_fused": 2.0 * Mc * w.H * w.dh * w.d}
    kinds = {}
    for r in records:
        k = kinds.setdefault(r["kind"], {"launches": 0, "total_ms": 0.0, "flops": 0.0})
        k["launches"] += 1
        k["total_ms"] += r["end_ms"] - r["start_ms"]
        k["flops"] += launch_flops.get(r["kind"], 0.0)
    for k in kinds.values():
        k["avg_us"] = 1e3 * k["total_ms"] / k["launches"]
    a_tf = kinds["attn"]["flops"] / (kinds["attn"]["total_ms"] * 1e-3) / 1e12
    peak_tf, peak_key = tensor_peak_for(peaks, kinds["attn"]["avg_us"] * 1e-6)
    sustained_tf = float(peaks.get("bf16_tflops_sustained", peak_tf))
    span_ms, exposed_ms = timeline_stats(records)  # the fused launch counts as GEMM time here
    if fused_tail is not None:
        exposed_ms += fused_tail
    value = whole_job_tflops(w.flops(), world, mean_ms)
    line = {
        "metric": "sliced TP attention block TFLOP/s at 1 GB300 (% BF16 peak); exposed shard-reduce time/layer",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) activations, N(0,1/fan_in) weights, bf16",
        "config": {"workload": w.name, "B": w.B, "S": w.S, "d": w.d, "H": w.H, "dh": w.dh, "P": w.P, "mu": w.mu,
                   "partials": w.partial, "schedule": schedule, "causal": True,
                   "l2": "flushed between steps (256 MiB write outside the step events)",
                   **({"plan": args.plan_result} if getattr(args, "plan_result", None) else {})},
        "pct_of_bf16_peak": round(100.0 * value / world / peak_tf, 2),
        "exposed_reduce_us_per_layer": round(1e3 * exposed_ms, 2),
        "exposed_reduce_frac": round(exposed_ms / span_ms, 4) if span_ms > 0 else None,
        "roofline": {
            "kernel": "attn_fwd_kernel (causal attention core)",
            "note": "achieved = causal attention flops (Q K^T and P V over the visible query-key pairs) of the "
                    "kernel's launches / their summed event durations",
            "bound": "tensor", "achieved": round(a_tf, 2), "peak": peak_tf, "unit": "TFLOP/s",
            "frac": round(a_tf / peak_tf, 4), "peak_source": f"{peak_src} {peak_key}",
            "avg_launch_us": round(kinds["attn"]["avg_us"], 2), "frac_of_sustained": round(a_tf / sustained_tf, 4),
            "flops_per_launch": float(core_flops_chunk), "traffic": ncu_traffic("attn", w.name, w.mu),
            "frac_of_mma_probe": round(a_tf / probe["tflops"], 4),
        },
        "tensor_probe": probe,
        "device": device_info(dev),
        "kernels": {k: {"launches": v["launches"], "avg_us": round(v["avg_us"], 2),
                        "tflops": round(v["flops"] / (v["total_ms"] * 1e-3) / 1e12, 1) if v["flops"] else None,
                        "share": round(v["total_ms"] / sum(x["total_ms"] for x in kinds.values()), 4)}
                    for k, v in kinds.items()},
        "gpu_launches": len(records),
        "e2e": {"value": round(whole_job_tflops(w.flops(), world, e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": w.M * w.d * 2, "d2h_bytes_per_step": w.M * w.d * 2,
                "ms_per_step": round(e2e_ms, 4),
                "mode": "pipelined: each step uploads its input from pinned host memory and downloads its result "
                        "on two copy streams, overlapping the neighbouring steps' compute (double-buffered); "
                        "each step also contains the 256 MiB L2 flush"},
        "e2e_serial": {"value": round(whole_job_tflops(w.flops(), world, e2e_serial_ms), 2), "unit": "TFLOP/s",
                       "ms_per_step": round(e2e_serial_ms, 4),
                       "mode": "upload, compute, download in order on one stream each step (L2 flush outside the events)"},
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        # one sequence at a time (sequences are independent; flops scale with sequences)
        f = {k: v.double().numpy() for k, v in t.items()}
        t0, n = time.perf_counter(), 0
        while n < w.B and (n == 0 or time.perf_counter() - t0 < args.cpu_seconds):
            rows = slice(n * w.S, (n + 1) * w.S)
            att.attn_fwd(f["X"][rows], f["Wqkv"], f["Wo"], w.S, w.H)
            n += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(w.flops() * n / w.B / dt / 1e12, 5), "unit": "TFLOP/s",
                                "cores": blas_threads(), "cpu": cpu_model(), "kind": "oracle",
                                "sample": f"fp64 attention oracle on {n} of {w.B} sequences ({dt:.1f} s)"}
    return line


# ---------------------------------------------------------- reference arm

def run_reference_attn(args, w):
    """The fp64 attention oracle as it stands on the host cores: one sequence per step."""
    from communication_overlap_domino_gb300 import workloads as wl
    import oracle.attention as att
    t = wl.generate_attn(w, seed=0)
    f = {k: v.double().numpy() for k, v in t.items()}
    X = f["X"][:w.S]
    for _ in range(args.warmup):
        att.attn_fwd(X, f["Wqkv"], f["Wo"], w.S, w.H)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        att.attn_fwd(X, f["Wqkv"], f["Wo"], w.S, w.H)
        times.append(time.perf_counter() - t0)
    mean_s = statistics.mean(times)
    value = w.flops() / w.B / mean_s / 1e12
    return {
        "impl": "reference",
        "metric": "sliced TP attention block TFLOP/s at 1 GB300 (% BF16 peak); exposed shard-reduce time/layer",
        "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * mean_s, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic: seeded bf16 values widened to fp64",
        "config": {"workload": w.name, "B": w.B, "S": w.S, "d": w.d, "H": w.H, "dh": w.dh, "P": w.P, "mu": w.mu,
                   "sequences_per_step": 1},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": blas_threads(),
                         "cpu": cpu_model(), "kind": "oracle",
                         "sample": f"fp64 attention oracle on 1 of {w.B} sequences per step"},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, w):
    """The fp64 CPU oracle as it stands, on the host cores: each step runs the
    oracle forward on a bounded row sample of the workload."""
    from communication_overlap_domino_gb300 import workloads as wl
    t = wl.generate(w, seed=0)
    budget_s = 150.0
    rows, dt, _ = oracle_row_sample(w, t, target_s=min(5.0, budget_s / max(1, args.steps + args.warmup)))
    f64 = {k: v.double().numpy() for k, v in t.items() if k not in ("X", "dY")}
    X = t["X"][:rows].double().numpy()
    dY = t["dY"][:rows].double().numpy() if w.bwd else None
    for _ in range(args.warmup):
        oracle_step(w, f64, X, dY)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, f64, X, dY)
        times.append(time.perf_counter() - t0)
    mean_s = statistics.mean(times)
    flops = (w.fwd_flops() + (w.bwd_flops() if w.bwd else 0)) * rows / w.M
    value = flops / mean_s / 1e12
    what = "forward+backward" if w.bwd else "forward"
    sample = f"fp64 oracle {what} on {rows} of {w.M} rows per step"
    return {
        "impl": "reference",
        "metric": "sliced TP-MLP layer TFLOP/s at 1 GB300 (% BF16 peak); exposed shard-reduce time/layer",
        "value": round(value, 5),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * mean_s, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded N(0,1) activations, N(0,0.02) weights, bf16 values widened to fp64",
        "config": {"workload": w.name, "M": w.M, "d": w.d, "F": w.F, "P": w.P, "mu": w.mu, "act": w.act,
                   "partials": w.partial, "out_slices": w.slices, "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": blas_threads(),
                         "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--mu", type=int, default=None)
    ap.add_argument("--schedule", choices=("streams", "serial", "fused"), default=None,
                    help="default: fused for the MLP workloads; for the attention block, with --mu not given "
                         "either, domino_attn_plan's mu and schedule (streams, its faster schedule)")
    ap.add_argument("--plan", action="store_true",
                    help="take mu and the schedule from domino_mlp_plan (domino_attn_plan for the attention "
                         "block; overrides --mu and --schedule)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ab-pairs", type=int, default=30,
                    help="alternating full / partials-only calls for the A/B measure of the reduction (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from communication_overlap_domino_gb300 import workloads as wl
    name = args.workload or wl.BENCH_WORKLOAD
    w = wl.ATTN_WORKLOADS[name] if name in wl.ATTN_WORKLOADS else wl.WORKLOADS[name]
    if args.mu is not None:
        w = w.with_(mu=args.mu)
    attention = name in wl.ATTN_WORKLOADS
    if attention and args.mu is None and args.schedule is None:
        args.plan = True  # the attention block runs at domino_attn_plan's mu unless told otherwise
    if args.schedule is None:
        args.schedule = "streams" if attention else "fused"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps((run_reference_attn if attention else run_reference)(args, w)), flush=True)
        return

    import __graft_entry__
    __graft_entry__.build()
    args.plan_result = None
    if args.plan:
        import torch
        from communication_overlap_domino_gb300 import binding as b
        torch.cuda.set_device(local_rank)
        if attention:
            args.plan_result = b.plan_attn(w.B, w.S, w.d, w.H, w.P, w.partial, dh=w.dh)
        else:
            args.plan_result = b.plan(w.M, w.d, w.F, w.P, w.act, w.partial, w.slices)
        w = w.with_(mu=args.plan_result["mu"])
        args.schedule = args.plan_result["schedule"]
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        line = (run_attn if attention else run_ours)(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
