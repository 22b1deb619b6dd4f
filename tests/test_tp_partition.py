"""The tensor-parallel partition of the sliced MLP on two CPU ranks (gloo).

On P GPUs the block shards one rank per shard: rank p holds A_p (the column
shard of A, or of Wg and Wu) and B_p (the matching row shard of B), computes its
row-parallel partial Z_{k,p,s} = act(X_k A_p) B_p[:, s] for each chunk k and
output slice s, and the sum over shards becomes an all-reduce of each (k, s)
piece, issued as soon as the piece exists so that it runs while the rank goes on
to the next chunk (the Domino page, "Domino: Eliminating Communication in LLM
Training via Generic Tensor Slicing and Overlapping", Abstract: independent
pieces whose communication overlaps the next piece's computation).

Here the ranks are gloo processes on the CPU, each partial comes from the fp64
oracle applied to the rank's own shard (a shard's partial is the plain block of
hidden width F/P), and every all-reduce is asynchronous: all pieces of chunk k
are in flight while chunk k+1 is computed, and they are waited for only at the
end.  The result must equal the unsharded oracle, and every rank must issue the
pieces in the same (chunk, slice) order -- collectives match by issue order.
"""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from communication_overlap_domino_gb300 import workloads as wl

WORLD = 2


def _piece_order(mu, S):
    return [(k, s) for k in range(mu) for s in range(S)]


def _rank(rank, world, port, w, seed, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        f = wl.to_float64(wl.generate(w, seed))
        cols = slice(rank * w.Fp, (rank + 1) * w.Fp)  # this rank's shard of the hidden units
        A_p = (f["Wg"][:, cols], f["Wu"][:, cols]) if w.act == "swiglu" else f["A"][:, cols]
        B_p = f["B"][cols]
        ds = w.d // w.slices
        in_flight, issued = [], []
        for k in range(w.mu):
            rows = slice(k * w.Mc, (k + 1) * w.Mc)
            for s in range(w.slices):
                sc = slice(s * ds, (s + 1) * ds)
                piece = torch.from_numpy(np.ascontiguousarray(oracle.mlp_fwd(f["X"][rows], A_p, B_p[:, sc], w.act)))
                in_flight.append((rows, sc, piece, dist.all_reduce(piece, async_op=True)))
                issued.append((k, s))
        Y = np.full((w.M, w.d), np.nan)
        for rows, sc, piece, work in in_flight:
            work.wait()
            Y[rows, sc] = piece.numpy()
        orders = [None] * world
        dist.all_gather_object(orders, issued)
        out.put((rank, Y, orders))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("w", [
    wl.Workload("tp_gelu", M=96, d=48, F=64, P=WORLD, mu=3, act="gelu", partial="f32", slices=2),
    wl.Workload("tp_swiglu", M=64, d=32, F=48, P=WORLD, mu=4, act="swiglu", partial="bf16", slices=1),
], ids=lambda w: w.name)
def test_one_shard_per_rank_all_reduce_per_piece(w):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + os.getpid() % 200 + (7 if w.act == "swiglu" else 0)
    procs = [ctx.Process(target=_rank, args=(r, WORLD, port, w, 41, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    f = wl.to_float64(wl.generate(w, 41))
    A = (f["Wg"], f["Wu"]) if w.act == "swiglu" else f["A"]
    ref = oracle.mlp_fwd(f["X"], A, f["B"], w.act)
    for rank, Y, orders in res:
        assert np.all(np.isfinite(Y)), f"rank {rank}: a piece was never received"
        assert oracle.max_rel_err(Y, ref) <= 1e-12, f"rank {rank}"
        assert all(o == _piece_order(w.mu, w.slices) for o in orders), "ranks issued the pieces in different orders"
