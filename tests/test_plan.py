"""Schedule selection (domino_mlp_plan, domino_attn_plan) on the host: the rules
stated in include/domino.h, checked with explicit hardware figures (no device
needed).

The rule: schedule FUSED when the fused cooperative forward can be launched,
else STREAMS; mu = the smallest power of two dividing M whose chunk of hidden
activations (M/mu * F * 2 bytes) fits in 9/10 of the L2, among the mu whose
chunk still has at least one paired GEMM1 tile per 2-CTA cluster; else the
largest such mu; else 1.
"""
import os

import pytest

from communication_overlap_domino_gb300 import binding as b
from communication_overlap_domino_gb300 import workloads as wl

GB300 = dict(num_sms=152, l2_bytes=126 * 2**20, fused_available=1)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(b.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return b.lib()


def plan_for(w, **hw):
    return b.plan(w.M, w.d, w.F, w.P, w.act, w.partial, w.slices, **{**GB300, **hw})


def test_plan_headline_workloads(lib):
    budget = 126 * 2**20 // 10 * 9
    # GPT-style: one chunk's H = 4096 * 10240 * 2 = 83.9 MB fits the budget at mu = 1
    p = plan_for(wl.WORKLOADS["gpt_gelu_fwd"])
    assert (p["mu"], p["schedule"], p["reason"]) == (1, "fused", "fits_l2")
    assert p["chunk_h_bytes"] == 4096 * 10240 * 2 <= budget
    # Llama-style: 8192 * 11008 * 2 = 180 MB does not fit; half of it (90 MB) does
    p = plan_for(wl.WORKLOADS["llama_swiglu_fwd"])
    assert (p["mu"], p["reason"]) == (2, "fits_l2")
    assert 8192 * 11008 * 2 > budget >= p["chunk_h_bytes"] == 4096 * 11008 * 2
    # large SwiGLU: 16384 * 13824 * 2 = 453 MB; a quarter (113 MB) fits
    p = plan_for(wl.WORKLOADS["large_swiglu_fwd"])
    assert (p["mu"], p["reason"]) == (4, "fits_l2")
    assert p["chunk_h_bytes"] == 4096 * 13824 * 2 <= budget < 2 * p["chunk_h_bytes"]


def test_plan_schedule_follows_fused_availability(lib):
    w = wl.WORKLOADS["llama_swiglu_fwd"]
    assert plan_for(w, fused_available=0)["schedule"] == "streams"
    assert plan_for(w, fused_available=0)["mu"] == plan_for(w)["mu"]


def test_plan_small_problem(lib):
    p = plan_for(wl.WORKLOADS["tiny_gelu_fwd"])  # 1 x 4 x 2 = 8 paired GEMM1 tiles < 76 clusters
    assert (p["mu"], p["reason"]) == (1, "small")
    assert p["gemm1_tiles_per_chunk"] == 8


def test_plan_largest_filling_when_nothing_fits(lib):
    # a tiny L2: no chunk fits, so the finest chunking that still fills the GPU
    p = b.plan(16384, 4096, 16384, 8, "gelu", "bf16", num_sms=152, l2_bytes=2**20, fused_available=1)
    assert p["reason"] == "largest_filling"
    mu = p["mu"]
    tiles = lambda m: -(-(16384 // m) // 256) * (2048 // 256) * 8
    assert tiles(mu) >= 76 and (16384 % (2 * mu) or tiles(2 * mu) < 76 or 2 * mu > 64)


def test_plan_respects_divisibility_and_piece_limit(lib):
    # M = 2 * 3075: only mu = 1 and 2 divide M; no chunk of H fits, so the largest of them
    p = b.plan(6150, 4096, 65536, 8, "gelu", "bf16", **GB300)
    assert (p["mu"], p["reason"]) == (2, "largest_filling")
    # out_slices caps mu * out_slices at DOMINO_MAX_PIECES (64)
    p = b.plan(1 << 20, 512, 1 << 16, 1, "gelu", "bf16", out_slices=32, **GB300)
    assert p["mu"] * 32 <= 64


@pytest.mark.parametrize("F", [2048, 4096, 8192, 16384, 32768, 65536])
def test_plan_monotone_in_hidden_width(lib, F):
    # a wider hidden layer never asks for fewer chunks
    mus = [b.plan(8192, 4096, f, 8, "swiglu", "bf16", **GB300)["mu"] for f in (F, 2 * F)]
    assert mus[0] <= mus[1]


@pytest.mark.parametrize("kw,status", [
    (dict(P=0), 1), (dict(F=2047), 2), (dict(d=516), 3),
])
def test_plan_rejects_invalid_problems(lib, kw, status):
    args = dict(M=4096, d=512, F=2048, P=2, act="gelu", partial="f32")
    args.update(kw)
    with pytest.raises(b.DominoError) as e:
        b.plan(**args, **GB300)
    assert e.value.status == status


# ------------------------------------------------------------ attention block
# domino_attn_plan: the same rule over whole-sequence chunks, with one chunk's Q|K|V (B/mu * S * 3 H dh * 2
# bytes) as the intermediate that must fit in 9/10 of the L2 and the Q|K|V projection's paired tiles as the
# filling test; the schedule is always STREAMS.

def attn_plan_for(w, **hw):
    return b.plan_attn(w.B, w.S, w.d, w.H, w.P, w.partial, dh=w.dh,
                       **{**dict(num_sms=GB300["num_sms"], l2_bytes=GB300["l2_bytes"]), **hw})


def test_attn_plan_workloads(lib):
    budget = 126 * 2**20 // 10 * 9
    # GPT-style: all 4 sequences' Q|K|V, 4096 * 3 * 2560 * 2 = 62.9 MB, fit at mu = 1
    p = attn_plan_for(wl.ATTN_WORKLOADS["gpt_attn_fwd"])
    assert (p["mu"], p["schedule"], p["reason"]) == (1, "streams", "fits_l2")
    assert p["chunk_qkv_bytes"] == 4096 * 3 * 2560 * 2 <= budget
    # 16 row blocks x 8 column blocks (3 * 5 heads * 128 = 1920 columns per shard) x 4 shards
    assert p["proj_tiles_per_chunk"] == 16 * 8 * 4
    # Llama-style: 8192 * 3 * 4096 * 2 = 201 MB does not fit; two sequences (101 MB) do
    p = attn_plan_for(wl.ATTN_WORKLOADS["llama_attn_fwd"])
    assert (p["mu"], p["schedule"], p["reason"]) == (2, "streams", "fits_l2")
    assert 8192 * 3 * 4096 * 2 > budget >= p["chunk_qkv_bytes"] == 4096 * 3 * 4096 * 2


def test_attn_plan_small_and_empty(lib):
    # 256 rows: 1 row block x 2 column blocks (384 columns) x 2 shards = 4 tiles < 76 clusters
    p = attn_plan_for(wl.ATTN_WORKLOADS["tiny_attn_fwd"])
    assert (p["mu"], p["reason"], p["proj_tiles_per_chunk"]) == (1, "small", 4)
    p = b.plan_attn(0, 1024, 2560, 20, 4, "f32", num_sms=152, l2_bytes=126 * 2**20)
    assert (p["mu"], p["reason"], p["chunk_qkv_bytes"]) == (1, "small", 0)


def test_attn_plan_largest_filling_and_divisibility(lib):
    # a tiny L2: nothing fits, so the finest whole-sequence chunking that still fills the GPU
    p = b.plan_attn(16, 2048, 4096, 32, 8, "bf16", num_sms=152, l2_bytes=2**20)
    tiles = lambda mu: -(-(16 // mu * 2048) // 256) * (3 * 4 * 128 // 256) * 8
    assert p["reason"] == "largest_filling"
    assert tiles(p["mu"]) >= 76 and (p["mu"] == 16 or tiles(2 * p["mu"]) < 76)
    # B = 6: only mu = 1 and 2 divide it
    p = b.plan_attn(6, 2048, 4096, 32, 8, "bf16", num_sms=152, l2_bytes=2**20)
    assert (p["mu"], p["reason"]) == (2, "largest_filling")


@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192])
def test_attn_plan_monotone_in_sequence_length(lib, S):
    # longer sequences never ask for fewer chunks
    mus = [b.plan_attn(8, s, 4096, 32, 8, "bf16", num_sms=152, l2_bytes=126 * 2**20)["mu"] for s in (S, 2 * S)]
    assert mus[0] <= mus[1]


@pytest.mark.parametrize("kw,status", [
    (dict(P=0), 1), (dict(H=21), 2), (dict(dh=64), 2), (dict(S=1000), 2), (dict(d=2564), 3),
])
def test_attn_plan_rejects_invalid_problems(lib, kw, status):
    args = dict(B=4, S=1024, d=2560, H=20, P=4, partial="f32")
    args.update(kw)
    with pytest.raises(b.DominoError) as e:
        b.plan_attn(**args, num_sms=152, l2_bytes=126 * 2**20)
    assert e.value.status == status
