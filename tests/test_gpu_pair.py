"""Both GEMM tilings of the separate-launch schedules vs the fp64 oracle, through
the C ABI (needs a GB300): paired-CTA 256x256 tiles (tcgen05 cta_group::2, the
default) and one-CTA 128x256 tiles (DOMINO_FLAG_ONE_CTA)."""
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


def _inputs(w, t):
    dev = torch.device("cuda:0")
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    return t["X"].to(dev), A_sh, B_sh


def _fwd(w, t, pair, schedule="serial"):
    X, A_sh, B_sh = _inputs(w, t)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, schedule, pair_cta=pair)
    ws = torch.zeros(b.workspace_size(desc), dtype=torch.uint8, device="cuda")
    Y = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                  schedule=schedule, workspace=ws, pair_cta=pair, timeout_ns=500_000_000)
    st = b.query_device_status(ws)
    assert st == 0, f"device status {b.STATUS.get(st)}: {b.lib().domino_last_error().decode()}"
    return Y


def _ref(w, t, rows=None):
    f = wl.to_float64(t)
    X = f["X"] if rows is None else f["X"][rows]
    A = (f["Wg"], f["Wu"]) if w.act == "swiglu" else f["A"]
    return oracle.mlp_fwd(X, A, f["B"], w.act)


def test_paired_and_one_cta_agree():
    w = wl.WORKLOADS["tiny_gelu_fwd"]
    t = wl.generate(w, 0)
    yp = _fwd(w, t, pair=True)
    err = oracle.max_rel_err(yp.double().cpu().numpy(), _ref(w, t))
    assert err <= TOL, err
    y1 = _fwd(w, t, pair=False)
    assert oracle.max_rel_err(yp.double().cpu().numpy(), y1.double().cpu().numpy()) <= TOL


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "identity"])
@pytest.mark.parametrize("partial", ["f32", "bf16"])
@pytest.mark.parametrize("pair", [True, False])
def test_pair_ragged(act, partial, pair):
    w = wl.Workload("ragged", M=600, d=336, F=984, P=3, mu=3, act=act, partial=partial, slices=2)
    t = wl.generate(w, 3)
    y = _fwd(w, t, pair=pair, schedule="streams")
    assert oracle.max_rel_err(y.double().cpu().numpy(), _ref(w, t)) <= TOL


def test_pair_llama_tail():
    w = wl.Workload("llama_tail", M=512, d=512, F=2752, P=2, mu=2, act="swiglu", partial="bf16")
    t = wl.generate(w, 4)
    y = _fwd(w, t, pair=True, schedule="streams")
    assert oracle.max_rel_err(y.double().cpu().numpy(), _ref(w, t)) <= TOL


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("pair", [True, False])
def test_pair_backward(act, pair):
    w = wl.Workload("pair_bwd", M=600, d=336, F=984, P=3, mu=3, act=act, partial="f32", slices=2, bwd=True)
    t = wl.generate(w, 8, with_dy=True)
    X, A_sh, B_sh = _inputs(w, t)
    dY = t["dY"].cuda()
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, "streams", pair_cta=pair)
    saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(b.workspace_size(desc, with_bwd=True), dtype=torch.uint8, device="cuda")
    b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, saved=saved,
              workspace=ws, pair_cta=pair, timeout_ns=500_000_000)
    dX, dA_sh, dB_sh = b.mlp_bwd(X, A_sh, B_sh, dY, saved, F=w.F, mu=w.mu, act=w.act, partial=w.partial,
                                 out_slices=w.slices, workspace=ws, pair_cta=pair, timeout_ns=500_000_000)
    assert b.query_device_status(ws) == 0
    dA, dB = b.unshard_grads(dA_sh, dB_sh, w.act)
    f = wl.to_float64(t)
    A = (f["Wg"], f["Wu"]) if w.act == "swiglu" else f["A"]
    ref = oracle.mlp_bwd(f["X"], A, f["B"], f["dY"], w.act)
    assert oracle.max_rel_err(dX.double().cpu().numpy(), ref["dX"]) <= TOL
    assert oracle.max_rel_err(dB.double().cpu().numpy(), ref["dB"]) <= TOL
    if w.act == "swiglu":
        assert oracle.max_rel_err(dA[0].double().cpu().numpy(), ref["dWg"]) <= TOL
        assert oracle.max_rel_err(dA[1].double().cpu().numpy(), ref["dWu"]) <= TOL
    else:
        assert oracle.max_rel_err(dA.double().cpu().numpy(), ref["dA"]) <= TOL


@pytest.mark.parametrize("name", ["gpt_gelu_fwd", "llama_swiglu_fwd"])
@pytest.mark.parametrize("pair", [True, False])
def test_pair_full_size(name, pair):
    w = wl.WORKLOADS[name]
    t = wl.generate(w, 0)
    y = _fwd(w, t, pair=pair, schedule="streams")
    rng = np.random.default_rng(0)
    rows = sorted(set(int(r) for k in range(w.mu) for r in
                      [k * w.Mc, k * w.Mc + w.Mc - 1, *(k * w.Mc + rng.integers(0, w.Mc, 4))]))
    assert oracle.max_rel_err(y[rows].double().cpu().numpy(), _ref(w, t, rows)) <= TOL
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("pair", [True, False])
def test_fused_both_tilings(act, pair):
    # odd number of 128-row blocks per chunk (Mc = 200 -> 2 blocks; M=1000, mu=2 -> 500 rows, 4 blocks with a
    # ragged last one; M=1152, mu=3 -> 384 rows, 3 blocks: the paired kernel's last pair has an empty half)
    for (M, mu) in ((600, 3), (1000, 2), (1152, 3)):
        w = wl.Workload("fused_tilings", M=M, d=336, F=984, P=3, mu=mu, act=act, partial="f32")
        t = wl.generate(w, 11)
        y = _fwd(w, t, pair=pair, schedule="fused")
        assert oracle.max_rel_err(y.double().cpu().numpy(), _ref(w, t)) <= TOL, (M, mu)
        ys = _fwd(w, t, pair=pair, schedule="streams")
        assert torch.equal(y, ys), "fused and stream schedules differ"
