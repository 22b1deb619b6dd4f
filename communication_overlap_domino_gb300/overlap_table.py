"""Pairwise overlap measurement: GEMM || shard-sum on one GB300.

The DHelix review page ("Hiding Communication Cost in Distributed LLM Training
via Micro-batch Co-execution", What carries the argument / Referee Report) rests
its scheduler on measured costs of operator pairs run together, and questions
whether those costs add up when the pair runs inside a longer schedule.  This
tool measures the same thing for the pair this library overlaps: a GEMM of
chunk k+1 and the shard-sum of chunk k.

For each workload it runs the layer twice through the C ABI with per-launch
CUDA events:
  * SERIAL schedule: every kernel runs alone (the isolated costs);
  * STREAMS schedule: the shard-sum of chunk k runs on a second stream beside
    GEMM1 of chunk k+1 (the overlapped costs);
and reports, per workload, each kernel's mean duration alone and overlapped,
the slowdown factors, the layer time, and the layer time the isolated costs
predict if overlap were free (sum of the GEMMs plus the shard-sum of the
last piece) -- the additivity the pages' scheduler assumes.

    python -m communication_overlap_domino_gb300.overlap_table [--steps N] [--workloads a,b]
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import binding as b
from . import workloads as wl


def _run(w, schedule, steps, A_sh, B_sh, X, Y, ws, flush):
    def call(timed):
        b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                  schedule=schedule, Y=Y, workspace=ws, kernel_times=timed)

    for _ in range(3):
        call(False)
    torch.cuda.synchronize()
    b.kernel_times_reset()
    evs = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call(True)
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    recs = b.kernel_times()
    layer_ms = statistics.mean(a.elapsed_time(c) for a, c in evs)
    by = {}
    for r in recs:
        by.setdefault((r["kind"], r["chunk"], r["slice"]), []).append(r["end_ms"] - r["start_ms"])
    return layer_ms, {k: statistics.mean(v) for k, v in by.items()}


def measure(w, steps=50):
    dev = torch.device("cuda", torch.cuda.current_device())
    t = wl.generate(w, 0)
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    X = t["X"].to(dev)
    Y = torch.empty((w.M, w.d), dtype=torch.bfloat16, device=dev)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, "streams")
    ws = torch.zeros(b.workspace_size(desc), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    lay_s, alone = _run(w, "serial", steps, A_sh, B_sh, X, Y, ws, flush)
    lay_o, over = _run(w, "streams", steps, A_sh, B_sh, X, Y, ws, flush)
    if b.query_device_status(ws) != 0:
        raise RuntimeError("device status not OK")
    rows = []
    for (kind, k, s), t_alone in sorted(alone.items()):
        t_over = over.get((kind, k, s))
        rows.append({"kernel": kind, "chunk": k, "slice": s, "alone_us": round(1e3 * t_alone, 1),
                     "overlapped_us": None if t_over is None else round(1e3 * t_over, 1),
                     "slowdown": None if t_over is None else round(t_over / t_alone, 3)})
    gemm_alone = sum(v for (kind, _, _), v in alone.items() if kind != "shard_sum")
    last_red = max((v for (kind, k, s), v in alone.items()
                    if kind == "shard_sum" and k == w.mu - 1 and s == w.slices - 1), default=0.0)
    predicted = gemm_alone + last_red
    return {"workload": w.name, "mu": w.mu, "layer_serial_us": round(1e3 * lay_s, 1),
            "layer_streams_us": round(1e3 * lay_o, 1),
            "layer_predicted_if_additive_us": round(1e3 * predicted, 1),
            "additivity_error": round(lay_o / predicted - 1.0, 4), "kernels": rows}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--workloads", default="gpt_gelu_fwd,llama_swiglu_fwd,large_swiglu_fwd")
    args = ap.parse_args()
    for name in args.workloads.split(","):
        print(json.dumps(measure(wl.WORKLOADS[name], args.steps)), flush=True)


if __name__ == "__main__":
    main()
