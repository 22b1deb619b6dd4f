"""Strand interleaving on one GB300: the forward of micro-batch a and the backward
of micro-batch b of the same layer, timed three ways (CUDA events, L2 flushed
before every step):

  sequential_fused    domino_mlp_fwd(a, FUSED) then domino_mlp_bwd(b)
  sequential_streams  domino_mlp_fwd(a, STREAMS) then domino_mlp_bwd(b)
  interleaved         domino_mlp_fwd_bwd_interleaved(a, b, STREAMS): strand b's
                      dH, then the chunks of the two strands alternate, the
                      shard-sums of each strand beside the other's GEMMs

The DHelix review page ("Hiding Communication Cost in Distributed LLM Training
via Micro-batch Co-execution") co-runs two strands so that one strand's
communication hides under the other's computation; this measures what that
buys against the tile-granular fused forward.

    python -m communication_overlap_domino_gb300.strands [--steps N] [--workloads a,b]
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import binding as b
from . import workloads as wl


def measure(w, steps=30):
    dev = torch.device("cuda", torch.cuda.current_device())
    ta, tb = wl.generate(w, 0, with_dy=True), wl.generate(w, 1, with_dy=True)
    A = (ta["Wg"].to(dev), ta["Wu"].to(dev)) if w.act == "swiglu" else ta["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, ta["B"].to(dev), w.P)
    Xa, Xb, dYb = ta["X"].to(dev), tb["X"].to(dev), tb["dY"].to(dev)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, "streams")
    saved_a = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=dev)
    saved_b = torch.zeros_like(saved_a)
    b.mlp_fwd(Xb, A_sh, B_sh, schedule="streams", saved=saved_b, **kw)
    Ya = torch.empty((w.M, w.d), dtype=torch.bfloat16, device=dev)
    dXb = torch.empty_like(Ya)
    dA = [torch.empty_like(a) for a in A_sh]
    dB = [torch.empty_like(x) for x in B_sh]
    ws_f = torch.zeros(b.workspace_size(desc), dtype=torch.uint8, device=dev)
    ws_b = torch.zeros(b.workspace_size(desc, with_bwd=True), dtype=torch.uint8, device=dev)
    ws_i = torch.zeros(b.interleaved_workspace_size(desc), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def sequential(fwd_schedule):
        def run():
            b.mlp_fwd(Xa, A_sh, B_sh, schedule=fwd_schedule, Y=Ya, saved=saved_a, workspace=ws_f, **kw)
            b.mlp_bwd(Xb, A_sh, B_sh, dYb, saved_b, schedule="streams", dX=dXb, dA_shards=dA, dB_shards=dB,
                      workspace=ws_b, **kw)
        return run

    def interleaved():
        b.mlp_fwd_bwd_interleaved(A_sh, B_sh, Xa, Xb, dYb, saved_b, schedule="streams", Ya=Ya, saved_a=saved_a,
                                  dXb=dXb, dA_shards=dA, dB_shards=dB, workspace=ws_i, **kw)

    flops = w.fwd_flops() + w.bwd_flops()
    out = {"workload": w.name, "M": w.M, "d": w.d, "F": w.F, "P": w.P, "mu": w.mu, "act": w.act, "steps": steps}
    for name, fn in (("sequential_fused", sequential("fused")), ("sequential_streams", sequential("streams")),
                     ("interleaved", interleaved)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(c) for a, c in evs)
        out[name] = {"us_per_step": round(1e3 * ms, 1), "tflops": round(flops / ms / 1e9, 1)}
    for ws in (ws_f, ws_b, ws_i):
        if b.query_device_status(ws) != 0:
            raise RuntimeError("device status not OK")
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--workloads", default="llama_swiglu_fwdbwd,gpt_gelu_fwd")
    args = ap.parse_args()
    for name in args.workloads.split(","):
        print(json.dumps(measure(wl.WORKLOADS[name].with_(bwd=True), args.steps)), flush=True)


if __name__ == "__main__":
    main()
