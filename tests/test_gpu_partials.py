"""domino_mlp_fwd_partials on the GB300: the row-parallel partials of every shard
without the sum over shards (the computation a tensor-parallel rank holds when
the all-reduce runs outside the library).

Bar: each partial Z_p = act(X A_p) B_p against the oracle's block with that
shard's weights (a shard's partial is the plain block of hidden width F/P),
max|Z - Z_ref| / max|Z_ref| <= 1e-2; the library's shard-sum of the partials
gives domino_mlp_fwd's Y bit for bit; a rank holding one shard (P = 1) computes
that shard's partial bit for bit; piece events let a consumer on another stream
start on each (chunk, slice) piece.
"""
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


def _setup(w, seed):
    t = wl.generate(w, seed)
    dev = torch.device("cuda:0")
    A = (t["Wg"].to(dev), t["Wu"].to(dev)) if w.act == "swiglu" else t["A"].to(dev)
    A_sh, B_sh = b.shard_weights(A, t["B"].to(dev), w.P)
    return t, t["X"].to(dev), A_sh, B_sh


def _shard_ref(w, f, p):
    cols = slice(p * w.Fp, (p + 1) * w.Fp)
    A = (f["Wg"][:, cols], f["Wu"][:, cols]) if w.act == "swiglu" else f["A"][:, cols]
    return oracle.mlp_fwd(f["X"], A, f["B"][cols], w.act)


CASES = [
    wl.Workload("partials_ragged", M=600, d=336, F=984, P=3, mu=3, act="gelu", partial="f32", slices=2),
    wl.Workload("partials_glu", M=1024, d=512, F=2752, P=2, mu=4, act="swiglu", partial="bf16", slices=2),
]


@pytest.mark.parametrize("schedule", ["serial", "streams", "fused"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_partials_match_oracle_and_sum_to_forward(w, schedule):
    t, X, A_sh, B_sh = _setup(w, 21)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule=schedule)
    Z = b.mlp_fwd_partials(X, A_sh, B_sh, **kw)
    Y = b.mlp_fwd(X, A_sh, B_sh, **kw)
    Ys = torch.empty_like(Y)
    b.shard_sum(Z, Ys)
    torch.cuda.synchronize()
    f = wl.to_float64(t)
    for p in range(w.P):
        err = oracle.max_rel_err(Z[p].double().cpu().numpy(), _shard_ref(w, f, p))
        assert err <= TOL, f"shard {p}: {err:.3e}"
    assert torch.equal(Ys, Y), "sum of the partials differs from the forward pass"


@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_partials_full_size_sum_to_forward(schedule):
    # the bench's configuration (the large SwiGLU layer, the "without" side of its A/B measure): the library's
    # shard-sum of the 8 partials gives the forward's Y bit for bit, and each partial on sampled rows matches the
    # oracle's block with that shard's weights
    w = wl.WORKLOADS["large_swiglu_fwd"]
    t, X, A_sh, B_sh = _setup(w, 22)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule=schedule)
    Z = b.mlp_fwd_partials(X, A_sh, B_sh, **kw)
    Y = b.mlp_fwd(X, A_sh, B_sh, **kw)
    Ys = torch.empty_like(Y)
    b.shard_sum(Z, Ys)
    torch.cuda.synchronize()
    assert torch.equal(Ys, Y), "sum of the partials differs from the forward pass"
    rows = torch.tensor([0, 127, 128, 255, 256, w.Mc - 1, w.Mc, w.M - 1])
    f = {k: v[rows].to(torch.float64).numpy() if k == "X" else v.to(torch.float64).numpy() for k, v in t.items()}
    for p in (0, w.P - 1):
        err = oracle.max_rel_err(Z[p][rows].double().cpu().numpy(), _shard_ref(w, f, p))
        assert err <= TOL, f"shard {p}: {err:.3e}"


@pytest.mark.parametrize("schedule", ["streams", "fused"])
def test_one_shard_rank_computes_its_partial(schedule):
    w = CASES[1]
    t, X, A_sh, B_sh = _setup(w, 22)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule=schedule)
    Z = b.mlp_fwd_partials(X, A_sh, B_sh, **kw)
    for p in range(w.P):  # rank p holds shard p alone: P = 1, hidden width F/P
        Zp = b.mlp_fwd_partials(X, [A_sh[p]], [B_sh[p]], **{**kw, "F": w.Fp})
        torch.cuda.synchronize()
        assert torch.equal(Zp[0], Z[p]), f"rank {p}"


def test_piece_events_let_a_consumer_start_per_piece():
    w = CASES[0]
    t, X, A_sh, B_sh = _setup(w, 23)
    kw = dict(F=w.F, mu=w.mu, act=w.act, partial=w.partial, out_slices=w.slices, schedule="streams")
    events = [torch.cuda.Event() for _ in range(w.mu * w.slices)]
    side = torch.cuda.Stream()
    Z = b.mlp_fwd_partials(X, A_sh, B_sh, piece_events=events, **kw)
    Y = torch.full((w.M, w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    ds = w.d // w.slices
    for k in range(w.mu):  # the consumer: per piece, wait for its event, then sum it on the side stream
        for s in range(w.slices):
            side.wait_event(events[k * w.slices + s])
            rows, cols = slice(k * w.Mc, (k + 1) * w.Mc), slice(s * ds, (s + 1) * ds)
            b.shard_sum([z[rows, cols] for z in Z], Y[rows, cols], stream=side)
    side.synchronize()
    torch.cuda.synchronize()
    ref = b.mlp_fwd(X, A_sh, B_sh, **kw)
    torch.cuda.synchronize()
    assert torch.equal(Y, ref)
