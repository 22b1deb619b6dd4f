"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300).

Bar: max|Y - Y_ref| / max|Y_ref| <= 1e-2 per output tensor (bf16 inputs, fp32
accumulation).  Small cases are compared element by element over the whole
output; the full-size workloads on rows sampled across every chunk (rows are
independent, so the oracle computes exactly those rows).
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


def _device_inputs(w, t):
    dev = torch.device("cuda:0")
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    return t["X"].to(dev), A_sh, B_sh


def _oracle_A(w, f64):
    return (f64["Wg"], f64["Wu"]) if w.act == "swiglu" else f64["A"]


def _run(w, t, schedule="streams", saved=None, Y=None):
    X, A_sh, B_sh = _device_inputs(w, t)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, schedule)
    ws = torch.zeros(b.workspace_size(desc), dtype=torch.uint8, device="cuda:0")
    Y = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices,
                  schedule=schedule, workspace=ws, saved=saved, Y=Y)
    status = b.query_device_status(ws)
    assert status == 0, f"device status {b.STATUS.get(status)}"
    return Y


def _check_full(w, seed=0, schedule="streams"):
    t = wl.generate(w, seed)
    Y = _run(w, t, schedule)
    f64 = wl.to_float64(t)
    ref = oracle.mlp_fwd(f64["X"], _oracle_A(w, f64), f64["B"], w.act)
    got = Y.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = oracle.max_rel_err(got, ref)
    assert err <= TOL, f"{w.name}: max rel err {err:.3e}"
    return err


# --------------------------------------------------------------- shard-sum

@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_shard_sum_parity(P, dtype):
    g = torch.Generator().manual_seed(100 + P)
    rows, cols, ld = 300, 136, 152
    parts_cpu = [torch.randn(rows, ld, generator=g).to(dtype) for _ in range(P)]
    parts = [z.cuda() for z in parts_cpu]
    Y = torch.full((rows, cols + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    b.shard_sum([z[:, :cols] for z in parts], Y[:, :cols])
    torch.cuda.synchronize()
    ref = oracle.shard_sum([z[:, :cols].double().numpy() for z in parts_cpu])
    got = Y[:, :cols].double().cpu().numpy()
    bound = 2.0 ** -8 * np.abs(ref) + P * 2.0 ** -22 * sum(np.abs(z[:, :cols].double().numpy()) for z in parts_cpu)
    assert np.all(np.abs(got - ref) <= bound + 1e-30)
    assert oracle.max_rel_err(got, ref) <= TOL
    assert torch.all(Y[:, cols:] == 7.0), "wrote outside the output columns"


# ---------------------------------------------------------- small workloads

@pytest.mark.parametrize("schedule", ["serial", "streams", "fused"])
def test_tiny_gelu_workload(schedule):
    _check_full(wl.WORKLOADS["tiny_gelu_fwd"], schedule=schedule)


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "identity"])
@pytest.mark.parametrize("partial", ["f32", "bf16"])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_ragged_shapes(act, partial, schedule):
    # chunk rows 200 (not a multiple of 128), F/P = 328 (N and K tails), d = 336
    # (K tail for GEMM1), two output slices of 168 columns (N tail), P = 3, mu = 3
    w = wl.Workload("ragged", M=600, d=336, F=984, P=3, mu=3, act=act, partial=partial, slices=2)
    _check_full(w, seed=3, schedule=schedule)


@pytest.mark.parametrize("h", [8, 40, 64, 96, 120, 0])
def test_swiglu_ragged_last_column_block(h):
    # F / P = 256 + h: the last SwiGLU column block holds h < 128 valid columns of gate and of up, the rest of
    # each 128-row weight box zero-filled (h = 0: no ragged block)
    w = wl.Workload(f"swiglu_ragged_{h}", M=512, d=256, F=2 * (256 + h), P=2, mu=2, act="swiglu", partial="bf16")
    _check_full(w, seed=11, schedule="fused")


@pytest.mark.parametrize("rows", [129, 200, 300, 700])
@pytest.mark.parametrize("act,partial", [("gelu", "f32"), ("swiglu", "bf16")])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_pair_row_tails(rows, act, partial, schedule):
    # the GEMMs run 256-row tiles on 2-CTA clusters, 128 rows per CTA: in the last tile of a chunk the
    # odd CTA holds 1 row (129), part of its block (200, 700) or lies wholly below the chunk (300).
    # Rows past M (a sentinel band after the output) must stay untouched.
    w = wl.Workload("pair_tail", M=2 * rows, d=512, F=768, P=2, mu=2, act=act, partial=partial)
    t = wl.generate(w, 11)
    Ybuf = torch.full((w.M + 64, w.d), 7.0, dtype=torch.bfloat16, device="cuda:0")
    Y = _run(w, t, schedule, Y=Ybuf[:w.M])
    f64 = wl.to_float64(t)
    ref = oracle.mlp_fwd(f64["X"], _oracle_A(w, f64), f64["B"], w.act)
    err = oracle.max_rel_err(Y.double().cpu().numpy(), ref)
    assert err <= TOL, f"rows {rows}: {err:.3e}"
    assert torch.all(Ybuf[w.M:] == 7.0), "wrote past the last row"


@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_llama_shard_width_tail(schedule):
    # F/P = 1376 as in the Llama-style workload (10.75 tiles of 128), small M and d
    w = wl.Workload("llama_tail", M=512, d=512, F=2752, P=2, mu=2, act="swiglu", partial="bf16")
    _check_full(w, seed=4, schedule=schedule)


@pytest.mark.parametrize("P,mu,S", [(1, 1, 1), (4, 4, 1), (2, 1, 4), (16, 2, 1), (3, 5, 1)])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_degenerate_slicings(P, mu, S, schedule):
    w = wl.Workload("degenerate", M=640, d=512, F=P * 128 * (3 if P == 3 else 1), P=P, mu=mu, act="gelu",
                    partial="f32", slices=S)
    _check_full(w, seed=5, schedule=schedule)


@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_single_row_chunks(schedule):
    # mu = M: every chunk is one row (each GEMM tile and shard-sum piece holds a single valid row)
    w = wl.Workload("single_rows", M=40, d=256, F=512, P=2, mu=40, act="gelu", partial="f32")
    _check_full(w, seed=9, schedule=schedule)


def test_empty_batch_leaves_output_untouched():
    w = wl.Workload("empty", M=0, d=512, F=1024, P=2, mu=1, act="gelu", partial="f32")
    t = wl.generate(w.with_(M=1))
    X, A_sh, B_sh = _device_inputs(w, t)
    Y = torch.full((1, 512), 3.0, dtype=torch.bfloat16, device="cuda")
    b.mlp_fwd(X[:0], A_sh, B_sh, F=w.F, mu=1, act="gelu", partial="f32", Y=Y[:0])
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0)


def test_deterministic_and_schedule_independent():
    w = wl.WORKLOADS["tiny_gelu_fwd"].with_(M=1024, mu=4)
    t = wl.generate(w, seed=6)
    y1 = _run(w, t, "streams").clone()
    y2 = _run(w, t, "streams").clone()
    y3 = _run(w, t, "serial").clone()
    assert torch.equal(y1, y2), "two runs differ"
    assert torch.equal(y1, y3), "serial and overlapped schedules differ"
    w8 = w.with_(mu=8)
    y4 = _run(w8, t, "streams")
    assert torch.equal(y1, y4), "result depends on mu"
    y5 = _run(w, t, "fused")
    assert torch.equal(y1, y5), "fused and stream schedules differ"
    y6 = _run(w8, t, "fused")
    assert torch.equal(y1, y6), "fused result depends on mu"


def test_fused_timeline_and_saved():
    w = wl.Workload("fused_saved", M=512, d=512, F=2048, P=4, mu=2, act="swiglu", partial="bf16")
    t = wl.generate(w, seed=10)
    X, A_sh, B_sh = _device_inputs(w, t)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial, w.slices, "fused")
    ws = torch.zeros(b.workspace_size(desc), dtype=torch.uint8, device="cuda")
    saved_f = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device="cuda")
    saved_s = torch.zeros_like(saved_f)
    yf = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, schedule="fused", workspace=ws,
                   saved=saved_f)
    tl = b.read_timeline(ws)
    assert tl["start_ns"] <= tl["gemm_end_ns"] and tl["start_ns"] <= tl["reduce_end_ns"]
    assert tl["reduce_end_ns"] - tl["start_ns"] < 10_000_000_000
    ys = b.mlp_fwd(X, A_sh, B_sh, F=w.F, mu=w.mu, act=w.act, partial=w.partial, schedule="streams", saved=saved_s)
    torch.cuda.synchronize()
    assert torch.equal(yf, ys)
    assert torch.equal(saved_f, saved_s), "fused schedule saved different pre-activations"
    assert b.query_device_status(ws) == 0


def test_saved_preactivations():
    w = wl.Workload("saved", M=256, d=512, F=2048, P=2, mu=2, act="swiglu", partial="bf16")
    t = wl.generate(w, seed=7)
    desc = b.make_desc(w.M, w.d, w.F, w.P, w.mu, w.act, w.partial)
    saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device="cuda")
    Y = _run(w, t, saved=saved)
    f64 = wl.to_float64(t)
    inter = oracle.mlp_fwd_intermediates(f64["X"], _oracle_A(w, f64), f64["B"], w.act)
    Fp = w.Fp
    # per shard: pre-activations [M, 2 Fp] (g | u), then H [M, Fp]
    blk = saved.view(torch.bfloat16).view(w.P, 3 * w.M * Fp)
    for p in range(w.P):
        cols = slice(p * Fp, (p + 1) * Fp)
        pre = blk[p, :2 * w.M * Fp].view(w.M, 2 * Fp).double().cpu().numpy()
        Hp = blk[p, 2 * w.M * Fp:].view(w.M, Fp).double().cpu().numpy()
        assert oracle.max_rel_err(pre[:, :Fp], inter["g"][:, cols]) <= TOL
        assert oracle.max_rel_err(pre[:, Fp:], inter["u"][:, cols]) <= TOL
        assert oracle.max_rel_err(Hp, inter["H"][:, cols]) <= TOL
    ref = inter["Y"]
    assert oracle.max_rel_err(Y.double().cpu().numpy(), ref) <= TOL


# ------------------------------------------------------- full-size workloads

# offsets within a chunk where one tile (128 rows per CTA, 256 per CTA pair, 512 per group of pairs) ends and
# the next begins
_TILE_EDGES = (0, 1, 127, 128, 255, 256, 511, 512)


def _sample_rows(w, per_chunk=64, seed=0):
    """Rows of every chunk for a sampled comparison: the tile edges, the chunk's last row and random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for k in range(w.mu):
        lo = k * w.Mc
        picked = {lo + o for o in _TILE_EDGES if o < w.Mc} | {lo + w.Mc - 1}
        while len(picked) < min(per_chunk, w.Mc):
            picked.add(lo + int(rng.integers(0, w.Mc)))
        rows += picked
    return sorted(int(r) for r in rows)


def _check_sampled(w, schedule="streams"):  # noqa: C901
    t = wl.generate(w, seed=0)
    Y = _run(w, t, schedule)
    rows = _sample_rows(w)
    f64 = {k: v[rows].to(torch.float64).numpy() if k == "X" else v.to(torch.float64).numpy() for k, v in t.items()}
    ref = oracle.mlp_fwd(f64["X"], _oracle_A(w, f64), f64["B"], w.act)
    got = Y[rows].double().cpu().numpy()
    err = oracle.max_rel_err(got, ref)
    assert err <= TOL, f"{w.name} mu={w.mu}: max rel err {err:.3e} on {len(rows)} sampled rows"
    # properties that hold at any size: finite everywhere, not all zero per chunk
    assert torch.isfinite(Y).all()
    for k in range(w.mu):
        assert Y[k * w.Mc:(k + 1) * w.Mc].abs().amax() > 0
    return err


@pytest.mark.parametrize("name", ["gpt_gelu_fwd", "llama_swiglu_fwd"])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_full_size_workload(name, schedule):
    _check_sampled(wl.WORKLOADS[name], schedule)


@pytest.mark.parametrize("mu", [1, 2, 4, 8])
@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_large_swiglu_mu_sweep(mu, schedule):
    _check_sampled(wl.WORKLOADS["large_swiglu_fwd"].with_(mu=mu), schedule)


@pytest.mark.parametrize("name,mus", [("large_swiglu_fwd", (4, 2)), ("gpt_gelu_fwd", (2, 1)),
                                      ("llama_swiglu_fwd", (4, 2))])
def test_full_size_bit_identical_across_schedules_and_mu(name, mus):
    # every output element is the same tiles' sums in the same order whatever the schedule and the chunking: the
    # whole output of the bench's configuration (FUSED at the first mu) equals STREAMS at that mu and FUSED at the
    # other bit for bit
    w = wl.WORKLOADS[name]
    t = wl.generate(w, 2)
    y_fused = _run(w.with_(mu=mus[0]), t, "fused")
    y_streams = _run(w.with_(mu=mus[0]), t, "streams")
    y_other_mu = _run(w.with_(mu=mus[1]), t, "fused")
    torch.cuda.synchronize()
    assert torch.equal(y_fused, y_streams), "fused and stream schedules differ"
    assert torch.equal(y_fused, y_other_mu), "result depends on mu"


# ------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_context_survives():
    """A device wait on a flag that nothing sets gives up after its limit, records
    DOMINO_ERR_TIMEOUT for the host, and the next call on the GPU still works."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert b.query_device_status(ws) == 0
    b.selftest_wait_timeout(ws, timeout_ns=50_000_000)  # 50 ms
    assert b.query_device_status(ws) == 6  # DOMINO_ERR_TIMEOUT
    assert "gave up" in b.lib().domino_last_error().decode()
    assert b.query_device_status(ws) == 0  # cleared by the read
    _check_full(wl.WORKLOADS["tiny_gelu_fwd"], schedule="fused")


@pytest.mark.parametrize("schedule", ["serial", "streams", "fused"])
def test_reserve_sms_leaves_results_unchanged(schedule):
    # the persistent grids shrink to (SMs - reserve_sms); every tile computes the same, so the result is equal
    w = wl.Workload("reserve", M=1000, d=336, F=1968, P=3, mu=2, act="swiglu", partial="bf16", slices=2)
    t = wl.generate(w, 19)
    X, A_sh, B_sh = _device_inputs(w, t)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule=schedule)
    y0 = b.mlp_fwd(X, A_sh, B_sh, **kw).clone()
    y1 = b.mlp_fwd(X, A_sh, B_sh, reserve_sms=16, **kw).clone()
    y2 = b.mlp_fwd(X, A_sh, B_sh, reserve_sms=torch.cuda.get_device_properties(0).multi_processor_count - 2, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(y0, y2)
    with pytest.raises(b.DominoError) as e:
        b.mlp_fwd(X, A_sh, B_sh, reserve_sms=torch.cuda.get_device_properties(0).multi_processor_count - 1, **kw)
    assert e.value.status == 1  # DOMINO_ERR_INVALID_ARG
