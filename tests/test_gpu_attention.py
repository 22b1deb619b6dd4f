"""The sliced tensor-parallel attention block (domino_attn_fwd) against the fp64
attention oracle, through the C ABI on the GB300.

Bar: max|Y - Y_ref| / max|Y_ref| <= 1e-2 (the block's own tolerance; Q, K, V, the
probabilities P and the attention output are rounded to bf16 on the GPU).  Small
problems are compared in full: one and several 128-query tiles per sequence
(the diagonal block and the blocks below it), one and several heads per shard,
one and several chunks, both partial precisions and both separate-launch
schedules.  At full size the oracle computes sampled sequences exactly (the
sequences are independent).
"""
import numpy as np
import pytest
import torch

import oracle.attention as att
from oracle import max_rel_err
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


def _run(w, t, schedule="streams", ws=None):
    dev = torch.device("cuda:0")
    qkv_sh, o_sh = b.shard_attn_weights(t["Wqkv"].to(dev), t["Wo"].to(dev), w.H, w.P)
    return b.attn_fwd(t["X"].to(dev), qkv_sh, o_sh, S=w.S, H=w.H, mu=w.mu, partial=w.partial, schedule=schedule,
                      workspace=ws)


def _f64(t):
    return {k: v.to(torch.float64).numpy() for k, v in t.items()}


@pytest.mark.parametrize("schedule", ["streams", "serial", "fused"])
@pytest.mark.parametrize("w", [
    wl.ATTN_WORKLOADS["tiny_attn_fwd"],
    wl.AttnWorkload("attn_4tiles", B=2, S=512, d=512, H=4, P=2, mu=2, partial="bf16"),
    wl.AttnWorkload("attn_one_shard", B=1, S=1024, d=256, H=1, P=1, mu=1, partial="f32"),
    wl.AttnWorkload("attn_3shards", B=3, S=256, d=384, H=6, P=3, mu=3, partial="f32"),
    # 5 query tiles per sequence (an odd count past one), 4 shards, 2 chunks: items of 1-5 key blocks dealt over
    # several rounds
    wl.AttnWorkload("attn_5tiles", B=2, S=640, d=512, H=4, P=4, mu=2, partial="bf16"),
    # 320 items of one key block each: every CTA runs several rounds and hands its output accumulator, row-sum
    # slots and Q slots over on every block
    wl.AttnWorkload("attn_many_short", B=160, S=128, d=256, H=2, P=2, mu=1, partial="f32"),
    # one work item in all: a grid of one CTA, one key block, no shard to sum with
    wl.AttnWorkload("attn_single_item", B=1, S=128, d=128, H=1, P=1, mu=1, partial="f32"),
], ids=lambda w: w.name if hasattr(w, "name") else w)
def test_attention_block_matches_oracle(w, schedule):
    t = wl.generate_attn(w, seed=5)
    Y = _run(w, t, schedule)
    torch.cuda.synchronize()
    f = _f64(t)
    ref = att.attn_fwd(f["X"], f["Wqkv"], f["Wo"], w.S, w.H)
    err = max_rel_err(Y.double().cpu().numpy(), ref)
    assert err <= TOL, f"{w.name}/{schedule}: {err:.3e}"


def test_attention_deterministic_and_schedule_independent():
    w = wl.AttnWorkload("attn_det", B=2, S=384, d=256, H=2, P=2, mu=2, partial="f32")
    t = wl.generate_attn(w, seed=6)
    a = _run(w, t, "streams")
    b2 = _run(w, t, "serial")
    c = _run(w.with_(mu=1), t, "streams")
    f = _run(w, t, "fused")  # each chunk's output projection and shard-sum in one cooperative launch
    torch.cuda.synchronize()
    assert torch.equal(a, b2) and torch.equal(a, c) and torch.equal(a, f)


def test_attention_device_status_and_empty_batch():
    w = wl.ATTN_WORKLOADS["tiny_attn_fwd"]
    t = wl.generate_attn(w, seed=7)
    desc = b.make_attn_desc(w.B, w.S, w.d, w.H, w.P, w.mu, w.partial)
    ws = torch.zeros(b.attn_workspace_size(desc), dtype=torch.uint8, device="cuda")
    _run(w, t, "streams", ws=ws)
    assert b.query_device_status(ws) == 0
    empty = b.make_attn_desc(0, w.S, w.d, w.H, w.P, 1, w.partial)
    assert b.lib().domino_attn_fwd(empty, None, None, None, None, None, 0, None) == 0


def _full_size_refs(name):
    # the workload's first and last sequence through the fp64 oracle, once per module
    w = wl.ATTN_WORKLOADS[name]
    t = wl.generate_attn(w, seed=0)
    f = _f64(t)
    refs = {}
    for seq in (0, w.B - 1):
        rows = slice(seq * w.S, (seq + 1) * w.S)
        refs[seq] = att.attn_fwd(f["X"][rows], f["Wqkv"], f["Wo"], w.S, w.H)
    return w, t, refs


@pytest.fixture(scope="module")
def gpt_full():
    return _full_size_refs("gpt_attn_fwd")


@pytest.fixture(scope="module")
def llama_full():
    return _full_size_refs("llama_attn_fwd")


def _check_sampled(w, t, refs, schedule):
    Y = _run(w, t, schedule).double().cpu().numpy()
    for seq, ref in refs.items():
        rows = slice(seq * w.S, (seq + 1) * w.S)
        err = max_rel_err(Y[rows], ref)
        assert err <= TOL, f"{w.name} mu {w.mu} {schedule}, sequence {seq}: {err:.3e}"
    assert np.isfinite(Y).all()


@pytest.mark.parametrize("mu", [1, 2])  # 1: the planned chunking the bench times; 2: the layer's MLP chunking
def test_gpt_attention_full_size_sampled(gpt_full, mu):
    w, t, refs = gpt_full
    _check_sampled(w.with_(mu=mu), t, refs, "streams")


@pytest.mark.parametrize("schedule", ["streams", "fused"])
@pytest.mark.parametrize("mu", [2, 4])  # 2: the planned chunking the bench times; 4: the layer's MLP chunking
def test_llama_attention_full_size_sampled(llama_full, schedule, mu):
    # 4 sequences of 2048 tokens, d 4096, 32 heads on 8 shards, bf16 partials: the first and the last sequence
    w, t, refs = llama_full
    _check_sampled(w.with_(mu=mu), t, refs, schedule)


@pytest.mark.parametrize("name,mus", [("gpt_attn_fwd", (1, 2)), ("llama_attn_fwd", (2, 4))])
def test_attention_full_size_independent_of_chunking(name, mus):
    # a sequence's output depends on nothing outside it, and every reduction runs in the same order whatever the
    # chunking: the whole output is bit-identical across mu
    w = wl.ATTN_WORKLOADS[name]
    t = wl.generate_attn(w, seed=1)
    a = _run(w.with_(mu=mus[0]), t)
    c = _run(w.with_(mu=mus[1]), t)
    torch.cuda.synchronize()
    assert torch.equal(a, c)
