"""domino_mlp_fwd_noalloc against domino_mlp_fwd (needs a GB300).

The no-allocation forward serves callers that cannot allocate device memory
while the layer runs (allocation-free real-time loops, hosts that own all device
memory, runtimes that forbid allocation after start-up): its scratch is a fixed
array inside the library instead of a caller workspace.  This file is collected
last so that a failure here leaves every other test already run; it passes in a
fresh process as well as after the other tests.
"""
import ctypes

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


def _inputs(w, seed):
    t = wl.generate(w, seed)
    A = (t["Wg"].cuda(), t["Wu"].cuda()) if w.act == "swiglu" else t["A"].cuda()
    A_sh, B_sh = b.shard_weights(A, t["B"].cuda(), w.P)
    return t["X"].cuda(), A_sh, B_sh, t


def _oracle_fwd(w, t):
    f = wl.to_float64(t)
    A = (f["Wg"], f["Wu"]) if w.act == "swiglu" else f["A"]
    return oracle.mlp_fwd(f["X"], A, f["B"], w.act)


def test_noalloc_matches_workspace_forward_on_two_calls_in_a_row():
    cases = [
        (wl.WORKLOADS["tiny_gelu_fwd"], 0),
        (wl.Workload("noalloc_swiglu", M=384, d=512, F=2752, P=2, mu=3, act="swiglu", partial="bf16", slices=2), 1),
    ]
    for w, seed in cases:
        desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices)
        assert b.workspace_size(desc) <= (32 << 20)
    results = []
    for w, seed in cases:  # two calls in a row, different problems, one shared scratch array
        X, A_sh, B_sh, t = _inputs(w, seed)
        Y = b.mlp_fwd_noalloc(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices)
        results.append((w, X, A_sh, B_sh, t, Y.clone()))
    st, header = b.mlp_fwd_noalloc_status()
    assert st == 0 and header % 256 == 0
    for w, X, A_sh, B_sh, t, Y in results:
        # the workspace forward with the same kernels in the same order: serial schedule, one-CTA tiles
        ref = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                        schedule="serial", pair_cta=False)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref), f"{w.name}: no-alloc and workspace forward differ"
        err = oracle.max_rel_err(Y.double().cpu().numpy(), _oracle_fwd(w, t))
        assert err <= TOL, f"{w.name}: no-alloc vs oracle {err:.3e}"


def test_noalloc_reports_a_device_timeout():
    """A bounded wait that runs out inside the fixed array's header is reported by
    domino_mlp_fwd_noalloc_status, cleared by the read, and the next call works."""
    w = wl.WORKLOADS["tiny_gelu_fwd"]
    X, A_sh, B_sh, t = _inputs(w, 2)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial)
    b.mlp_fwd_noalloc(X, A_sh, B_sh, **kw)
    st, header = b.mlp_fwd_noalloc_status()
    assert st == 0 and header != 0
    # the self-test wait records into the status words of the workspace it is given: here the header
    assert b.lib().domino_selftest_wait_timeout(header, 50_000_000, None) == 0
    st, _ = b.mlp_fwd_noalloc_status()
    assert st == 6, b.STATUS.get(st)  # DOMINO_ERR_TIMEOUT
    assert "gave up" in b.lib().domino_last_error().decode()
    assert b.mlp_fwd_noalloc_status()[0] == 0  # cleared by the read
    Y = b.mlp_fwd_noalloc(X, A_sh, B_sh, **kw)
    assert b.mlp_fwd_noalloc_status()[0] == 0
    assert oracle.max_rel_err(Y.double().cpu().numpy(), _oracle_fwd(w, t)) <= TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = wl.WORKLOADS["gpt_gelu_fwd"]
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial)
    assert b.workspace_size(desc) > (32 << 20)
    arr = b._ptr_array([0x20000] * w.P)
    st = b.lib().domino_mlp_fwd_noalloc(ctypes.byref(desc), 0x30000, arr, arr, 0x40000, None)
    assert st == 4  # DOMINO_ERR_WORKSPACE
    assert "scratch" in b.lib().domino_last_error().decode()
