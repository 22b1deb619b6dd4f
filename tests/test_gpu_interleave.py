"""Strand interleaving (domino_mlp_fwd_bwd_interleaved) on the GB300: the forward
of strand a and the backward of strand b in one call give bit-for-bit the
results of a separate domino_mlp_fwd(a) and domino_mlp_bwd(b), and each output
matches the fp64 oracle (max|g - g_ref| / max|g_ref| <= 1e-2 per tensor)."""
import pytest
import torch

import oracle
from communication_overlap_domino_gb300 import binding as b
from communication_overlap_domino_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _strands(w):
    dev = torch.device("cuda:0")
    ta, tb = wl.generate(w, 31, with_dy=True), wl.generate(w, 32, with_dy=True)
    A = (ta["Wg"].to(dev), ta["Wu"].to(dev)) if w.act == "swiglu" else ta["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, ta["B"].to(dev), w.P)
    return A_sh, B_sh, ta["X"].to(dev), tb["X"].to(dev), tb["dY"].to(dev), ta, tb


@pytest.mark.parametrize("schedule", ["streams", "serial"])
@pytest.mark.parametrize("w", [
    wl.Workload("interleave_ragged", M=600, d=336, F=984, P=3, mu=3, act="gelu", partial="f32", slices=2, bwd=True),
    wl.Workload("interleave_glu", M=1024, d=512, F=2752, P=2, mu=4, act="swiglu", partial="bf16", bwd=True),
], ids=lambda w: w.name if isinstance(w, wl.Workload) else w)
def test_interleaved_equals_separate_calls(w, schedule):
    A_sh, B_sh, Xa, Xb, dYb, ta, tb = _strands(w)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, schedule)
    saved_b = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=Xa.device)
    b.mlp_fwd(Xb, A_sh, B_sh, schedule="streams", saved=saved_b, **kw)
    # separate calls
    saved_a_ref = torch.zeros_like(saved_b)
    Ya_ref = b.mlp_fwd(Xa, A_sh, B_sh, schedule="streams", saved=saved_a_ref, **kw)
    dXb_ref, dA_ref, dB_ref = b.mlp_bwd(Xb, A_sh, B_sh, dYb, saved_b, schedule="streams", **kw)
    # one interleaved call
    saved_a = torch.zeros_like(saved_b)
    ws = torch.zeros(b.interleaved_workspace_size(desc), dtype=torch.uint8, device=Xa.device)
    Ya, dXb, dA, dB = b.mlp_fwd_bwd_interleaved(A_sh, B_sh, Xa, Xb, dYb, saved_b, schedule=schedule,
                                                saved_a=saved_a, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert b.query_device_status(ws) == 0
    assert torch.equal(Ya, Ya_ref) and torch.equal(saved_a, saved_a_ref) and torch.equal(dXb, dXb_ref)
    assert all(torch.equal(x, y) for x, y in zip(dA, dA_ref)) and all(torch.equal(x, y) for x, y in zip(dB, dB_ref))
    # against the oracle: strand a's forward, strand b's backward (weights are strand a's)
    fa, fb = wl.to_float64(ta), wl.to_float64(tb)
    A = (fa["Wg"], fa["Wu"]) if w.act == "swiglu" else fa["A"]
    f64 = lambda x: x.double().cpu().numpy()  # noqa: E731
    errs = {"Ya": oracle.max_rel_err(f64(Ya), oracle.mlp_fwd(fa["X"], A, fa["B"], w.act))}
    ref = oracle.mlp_bwd(fb["X"], A, fa["B"], fb["dY"], w.act)
    dA_full, dB_full = b.unshard_grads(dA, dB, w.act)
    errs["dXb"] = oracle.max_rel_err(f64(dXb), ref["dX"])
    errs["dB"] = oracle.max_rel_err(f64(dB_full), ref["dB"])
    if w.act == "swiglu":
        errs["dWg"] = oracle.max_rel_err(f64(dA_full[0]), ref["dWg"])
        errs["dWu"] = oracle.max_rel_err(f64(dA_full[1]), ref["dWu"])
    else:
        errs["dA"] = oracle.max_rel_err(f64(dA_full), ref["dA"])
    assert all(v <= 1e-2 for v in errs.values()), errs


@pytest.mark.parametrize("schedule", ["streams", "serial"])
def test_interleaved_full_size_equals_separate_calls(schedule):
    # the Llama-style layer at full size (8192 tokens, d 4096, F 11008, P 8, mu 4): every output of the one
    # interleaved call bit for bit that of the separate forward and backward calls (whose own parity with the
    # oracle is checked at this size on sampled rows and hidden units)
    w = wl.WORKLOADS["llama_swiglu_fwdbwd"]
    A_sh, B_sh, Xa, Xb, dYb, _, _ = _strands(w)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, schedule)
    saved_b = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=Xa.device)
    b.mlp_fwd(Xb, A_sh, B_sh, schedule="streams", saved=saved_b, **kw)
    saved_a_ref = torch.zeros_like(saved_b)
    Ya_ref = b.mlp_fwd(Xa, A_sh, B_sh, schedule="streams", saved=saved_a_ref, **kw)
    dXb_ref, dA_ref, dB_ref = b.mlp_bwd(Xb, A_sh, B_sh, dYb, saved_b, schedule="streams", **kw)
    saved_a = torch.zeros_like(saved_b)
    ws = torch.zeros(b.interleaved_workspace_size(desc), dtype=torch.uint8, device=Xa.device)
    Ya, dXb, dA, dB = b.mlp_fwd_bwd_interleaved(A_sh, B_sh, Xa, Xb, dYb, saved_b, schedule=schedule,
                                                saved_a=saved_a, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert b.query_device_status(ws) == 0
    assert torch.equal(Ya, Ya_ref) and torch.equal(saved_a, saved_a_ref) and torch.equal(dXb, dXb_ref)
    assert all(torch.equal(x, y) for x, y in zip(dA, dA_ref)) and all(torch.equal(x, y) for x, y in zip(dB, dB_ref))
    assert torch.isfinite(Ya).all() and torch.isfinite(dXb).all()
