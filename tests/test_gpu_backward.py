"""Backward pass of the sliced MLP vs the fp64 oracle, through the C ABI (GB300).

Bar per output tensor (dX, dA or dWg/dWu, dB): max|g - g_ref| / max|g_ref| <= 1e-2.
Small problems are compared in full.  At full size (the Llama-style fwd+bwd
workload) dX is checked on rows sampled from every chunk (rows of dX depend only
on the same rows of X and dY), and the weight gradients on sampled hidden units:
the columns of dWg, dWu and the rows of dWd that belong to a set of hidden units
depend only on those units' weights, so the oracle computes them exactly from the
column-restricted problem.
"""
import numpy as np
import pytest
import torch

import oracle
from communication_overlap_domino_gb300 import binding as b
from communication_overlap_domino_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run_fwd_bwd(w, t, schedule="streams"):
    dev = torch.device("cuda:0")
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    X, dY = t["X"].to(dev), t["dY"].to(dev)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, schedule)
    saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=dev)
    ws = torch.zeros(b.workspace_size(desc, with_bwd=True), dtype=torch.uint8, device=dev)
    Y = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                  schedule=schedule, saved=saved, workspace=ws)
    dX, dA_sh, dB_sh = b.mlp_bwd(X, A_sh, B_sh, dY, saved, F=w.F, mu=w.mu, act=w.act, partial=w.partial,
                                 out_slices=w.slices, schedule=schedule, workspace=ws)
    assert b.query_device_status(ws) == 0
    dA, dB = b.unshard_grads(dA_sh, dB_sh, w.act)
    return Y, dX, dA, dB


def _f64(t):
    return t.double().cpu().numpy()


def _check_full(w, seed, schedule="streams"):
    t = wl.generate(w, seed, with_dy=True)
    Y, dX, dA, dB = _run_fwd_bwd(w, t, schedule)
    f = wl.to_float64(t)
    A = (f["Wg"], f["Wu"]) if w.act == "swiglu" else f["A"]
    ref = oracle.mlp_bwd(f["X"], A, f["B"], f["dY"], w.act)
    errs = {"Y": oracle.max_rel_err(_f64(Y), oracle.mlp_fwd(f["X"], A, f["B"], w.act)),
            "dX": oracle.max_rel_err(_f64(dX), ref["dX"]),
            "dB": oracle.max_rel_err(_f64(dB), ref["dB"])}
    if w.act == "swiglu":
        errs["dWg"] = oracle.max_rel_err(_f64(dA[0]), ref["dWg"])
        errs["dWu"] = oracle.max_rel_err(_f64(dA[1]), ref["dWu"])
    else:
        errs["dA"] = oracle.max_rel_err(_f64(dA), ref["dA"])
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"{w.name}: {errs}"
    return errs


def test_tiny_backward():
    _check_full(wl.WORKLOADS["tiny_gelu_fwd"].with_(bwd=True), seed=0)


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "identity"])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_backward_ragged(act, schedule):
    w = wl.Workload("ragged_bwd", M=600, d=336, F=984, P=3, mu=3, act=act, partial="f32", slices=2, bwd=True)
    _check_full(w, seed=8, schedule=schedule)


@pytest.mark.parametrize("act,partial", [("swiglu", "bf16"), ("gelu", "f32")])
def test_fused_backward_equals_streams(act, partial):
    # the FUSED backward computes the partial input gradients of every chunk and their shard-sum in one
    # cooperative launch: the same tiles, K order and shard order as the per-chunk launches, so bit-equal
    w = wl.Workload("fused_bwd", M=1000, d=336, F=1968, P=3, mu=2, act=act, partial=partial, bwd=True)
    t = wl.generate(w, 17, with_dy=True)
    ref = _run_fwd_bwd(w, t, "streams")
    got = _run_fwd_bwd(w, t, "fused")
    names = ("Y", "dX")
    for n, a, b2 in zip(names, got[:2], ref[:2]):
        assert torch.equal(a, b2), f"{n} differs between the fused and the stream schedules"
    ga = got[2] if isinstance(got[2], tuple) else (got[2],)
    ra = ref[2] if isinstance(ref[2], tuple) else (ref[2],)
    assert all(torch.equal(a, b2) for a, b2 in zip(ga, ra)) and torch.equal(got[3], ref[3])


def test_llama_fwdbwd_full_size_fused_equals_streams():
    # the bench's fwd+bwd configuration at full size (8192 tokens, d 4096, F 11008, P 8, mu 4): the FUSED forward
    # and backward against the per-chunk launches, every output bit for bit (the graded, column-ordered last row
    # group of the fused launches included)
    w = wl.WORKLOADS["llama_swiglu_fwdbwd"]
    t = wl.generate(w, 3, with_dy=True)
    ref = _run_fwd_bwd(w, t, "streams")
    got = _run_fwd_bwd(w, t, "fused")
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref[0]), "Y differs"
    assert torch.equal(got[1], ref[1]), "dX differs"
    assert all(torch.equal(a, c) for a, c in zip(got[2], ref[2])), "dA differs"
    assert torch.equal(got[3], ref[3]), "dB differs"


@pytest.mark.parametrize("schedule", ["serial", "fused"])
def test_backward_llama_tail_bf16_partials(schedule):
    w = wl.Workload("llama_tail_bwd", M=512, d=512, F=2752, P=2, mu=2, act="swiglu", partial="bf16", bwd=True)
    _check_full(w, seed=9, schedule=schedule)


def test_backward_partial_row_group():
    # dH runs once over all M with its tiles in row groups of one chunk: chunk rows 640 -> groups of 3
    # 256-row blocks over 5 blocks, so the last group is partial; F_p = 1376 leaves a 96-column tile
    w = wl.Workload("group_tail_bwd", M=1280, d=512, F=2752, P=2, mu=2, act="swiglu", partial="bf16", bwd=True)
    _check_full(w, seed=13)
    _check_full(w.with_(act="gelu", partial="f32"), seed=14)


@pytest.mark.parametrize("rows", [129, 300, 700])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_backward_pair_row_tails(rows, schedule):
    # 256-row tiles on 2-CTA clusters: the last tile's odd CTA holds 1 row (129), lies wholly below the
    # chunk (300) or holds part of its block (700); the dH and weight-gradient launches over all M then
    # end on a ragged block too
    w = wl.Workload("pair_tail_bwd", M=2 * rows, d=512, F=768, P=2, mu=2, act="swiglu", partial="bf16", bwd=True)
    _check_full(w, seed=15, schedule=schedule)


def test_backward_empty_batch_zeroes_weight_grads():
    w = wl.Workload("empty_bwd", M=1, d=512, F=1024, P=2, mu=1, act="swiglu", partial="bf16", bwd=True)
    t = wl.generate(w, 0, with_dy=True)
    A_sh, B_sh = b.shard_weights((t["Wg"].cuda(), t["Wu"].cuda()), t["B"].cuda(), w.P)
    dA = [torch.full_like(a, 5.0) for a in A_sh]
    dB = [torch.full_like(x, 5.0) for x in B_sh]
    X = t["X"].cuda()[:0]
    b.mlp_bwd(X, A_sh, B_sh, X, X, F=w.F, mu=1, act="swiglu", partial="bf16", dX=X, dA_shards=dA, dB_shards=dB)
    torch.cuda.synchronize()
    assert all(torch.all(a == 0) for a in dA) and all(torch.all(x == 0) for x in dB)


@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_llama_fwdbwd_full_size_sampled(schedule):
    w = wl.WORKLOADS["llama_swiglu_fwdbwd"]
    t = wl.generate(w, 0, with_dy=True)
    Y, dX, dA, dB = _run_fwd_bwd(w, t, schedule)
    rng = np.random.default_rng(0)
    # 64 rows of every chunk: the tile edges (128-row CTA blocks, 256-row pair tiles), the chunk's last
    # row and random rows
    rows = set()
    for k in range(w.mu):
        lo = k * w.Mc
        chunk = {lo + o for o in (0, 1, 127, 128, 255, 256, 511, 512) if o < w.Mc} | {lo + w.Mc - 1}
        while len(chunk) < 64:
            chunk.add(lo + int(rng.integers(0, w.Mc)))
        rows |= chunk
    rows = sorted(rows)
    Xr = t["X"][rows].double().numpy()
    dYr = t["dY"][rows].double().numpy()
    Wg, Wu, Wd = (t[k].double().numpy() for k in ("Wg", "Wu", "B"))
    ref_rows = oracle.mlp_bwd(Xr, (Wg, Wu), Wd, dYr, "swiglu")
    assert oracle.max_rel_err(_f64(dX[rows]), ref_rows["dX"]) <= TOL
    assert oracle.max_rel_err(_f64(Y[rows]), oracle.mlp_fwd(Xr, (Wg, Wu), Wd, "swiglu")) <= TOL
    # 10 hidden units of every shard: the column-tile edges (256-wide N tiles of dH, 64-deep K blocks of
    # dX), the shard's last unit (the N and K tails) and random units
    units = set()
    for p in range(w.P):
        lo = p * w.Fp
        shard = {lo + j for j in (0, 63, 64, 255, 256, 1279, 1280, w.Fp - 1) if j < w.Fp}
        while len(shard) < 10:
            shard.add(lo + int(rng.integers(0, w.Fp)))
        units |= shard
    units = sorted(units)
    ref_cols = oracle.mlp_bwd(t["X"].double().numpy(), (Wg[:, units], Wu[:, units]), Wd[units],
                              t["dY"].double().numpy(), "swiglu")
    assert oracle.max_rel_err(_f64(dA[0][:, units]), ref_cols["dWg"]) <= TOL
    assert oracle.max_rel_err(_f64(dA[1][:, units]), ref_cols["dWu"]) <= TOL
    assert oracle.max_rel_err(_f64(dB[units]), ref_cols["dB"]) <= TOL
    for g in (dX, dA[0], dA[1], dB):
        assert torch.isfinite(g).all()


def test_fused_backward_with_reserved_sms():
    # the cooperative dX launch on fewer clusters (reserve_sms) gives the same gradients
    w = wl.Workload("reserve_bwd", M=1000, d=336, F=1968, P=3, mu=2, act="swiglu", partial="bf16", bwd=True)
    t = wl.generate(w, 23, with_dy=True)
    dev = torch.device("cuda:0")
    A_sh, B_sh = b.shard_weights((t["Wg"].to(dev), t["Wu"].to(dev)), t["B"].to(dev), w.P)
    X, dY = t["X"].to(dev), t["dY"].to(dev)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, schedule="fused")
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, 1, "fused")
    saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=dev)
    b.mlp_fwd(X, A_sh, B_sh, saved=saved, **kw)
    g0 = b.mlp_bwd(X, A_sh, B_sh, dY, saved, **kw)
    g1 = b.mlp_bwd(X, A_sh, B_sh, dY, saved, reserve_sms=40, **kw)
    torch.cuda.synchronize()
    assert torch.equal(g0[0], g1[0])
    assert all(torch.equal(a, c) for a, c in zip(g0[1], g1[1])) and all(torch.equal(a, c) for a, c in zip(g0[2], g1[2]))
