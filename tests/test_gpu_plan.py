"""domino_mlp_plan and domino_attn_plan on the GB300 itself: the hardware
figures come from the device, and the planned configurations run and match the
oracles."""
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


def test_plan_reads_the_device():
    props = torch.cuda.get_device_properties(0)
    w = wl.WORKLOADS["llama_swiglu_fwd"]
    p = b.plan(w.M, w.d, w.F, w.P, w.act, w.partial, w.slices)
    explicit = b.plan(w.M, w.d, w.F, w.P, w.act, w.partial, w.slices, num_sms=props.multi_processor_count,
                      l2_bytes=props.L2_cache_size, fused_available=1)
    assert p == explicit
    assert p["l2_budget_bytes"] == props.L2_cache_size // 10 * 9
    assert w.M % p["mu"] == 0 and p["schedule"] == "fused"


def test_planned_configuration_runs():
    w0 = wl.Workload("plan_small", M=2048, d=1024, F=4096, P=4, mu=1, act="gelu", partial="f32")
    p = b.plan(w0.M, w0.d, w0.F, w0.P, w0.act, w0.partial, num_sms=16, l2_bytes=1 << 20, fused_available=1)
    assert p["mu"] > 1  # the small L2 forces chunking
    w = w0.with_(mu=p["mu"])
    t = wl.generate(w, 21)
    dev = torch.device("cuda:0")
    A_sh, B_sh = b.shard_weights(t["A"].to(dev), t["B"].to(dev), w.P)
    Y = b.mlp_fwd(t["X"].to(dev), A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, schedule=p["schedule"])
    f = wl.to_float64(t)
    err = oracle.max_rel_err(Y.double().cpu().numpy(), oracle.mlp_fwd(f["X"], f["A"], f["B"], w.act))
    assert err <= 1e-2


def test_attn_plan_reads_the_device():
    props = torch.cuda.get_device_properties(0)
    w = wl.ATTN_WORKLOADS["llama_attn_fwd"]
    p = b.plan_attn(w.B, w.S, w.d, w.H, w.P, w.partial)
    explicit = b.plan_attn(w.B, w.S, w.d, w.H, w.P, w.partial, num_sms=props.multi_processor_count,
                           l2_bytes=props.L2_cache_size)
    assert p == explicit
    assert p["l2_budget_bytes"] == props.L2_cache_size // 10 * 9
    assert w.B % p["mu"] == 0 and p["schedule"] == "streams"


def test_attn_planned_configuration_runs():
    import oracle.attention as att
    w0 = wl.AttnWorkload("attn_plan_small", B=4, S=512, d=512, H=4, P=2, mu=1, partial="f32")
    p = b.plan_attn(w0.B, w0.S, w0.d, w0.H, w0.P, w0.partial, num_sms=16, l2_bytes=1 << 20)
    assert p["mu"] > 1  # the small L2 forces chunking
    w = w0.with_(mu=p["mu"])
    t = wl.generate_attn(w, seed=23)
    dev = torch.device("cuda:0")
    qkv_sh, o_sh = b.shard_attn_weights(t["Wqkv"].to(dev), t["Wo"].to(dev), w.H, w.P)
    Y = b.attn_fwd(t["X"].to(dev), qkv_sh, o_sh, S=w.S, H=w.H, mu=w.mu, partial=w.partial, schedule=p["schedule"])
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    err = oracle.max_rel_err(Y.double().cpu().numpy(), att.attn_fwd(f["X"], f["Wqkv"], f["Wo"], w.S, w.H))
    assert err <= 1e-2
