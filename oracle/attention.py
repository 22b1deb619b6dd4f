"""Oracle for the sliced tensor-parallel attention block: plain, slow, fp64, CPU.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module; it
is used by the tests and the benchmark's CPU-baseline leg.  It shares no code
with the CUDA path.

What it computes
----------------
The Domino page ("Domino: Eliminating Communication in LLM Training via Generic
Tensor Slicing and Overlapping", Abstract) slices a whole transformer layer, of
which this is the attention half, the same way as the MLP: independent pieces
whose communication overlaps the next piece's computation.  The tensor-parallel
split is the Megatron-LM one (titles under "Builds on" on the Domino page): the
query/key/value projection is split by heads (column-parallel), the output
projection by the matching rows (row-parallel), and the sum over shards of the
row-parallel partials is the unsharded product.  The oracle is the plain
*unsharded* block in float64, causal multi-head self-attention without biases:

    Q | K | V = X Wqkv                      (X: B sequences of S tokens, [B S, d])
    O_h       = softmax(Q_h K_h^T / sqrt(dh) + causal mask) V_h    per sequence, head h
    Y         = [O_0 | ... | O_{H-1}] Wo

Wqkv is [d, 3 H dh] with the columns of all query heads, then all key heads,
then all value heads (head h: columns h dh .. (h+1) dh of each block); Wo is
[H dh, d].  The causal mask lets token t attend to tokens 0..t of its own
sequence.  ``attn_fwd_sharded`` writes the slicing out (sequence chunks, head
shards, partial outputs summed in shard order); it exists only so the tests can
check the slicing invariants against the unsharded form.

Pins: ``tests/oracle_pins.py`` checks these functions against brute-force scalar
loops, closed forms (uniform attention gives prefix means; one-token sequences
make attention the identity), causality and the slicing invariants;
``tests/test_oracle_mutations.py`` plants mistakes here and checks the pins
catch them.
"""
from __future__ import annotations

import math
from typing import Dict

import numpy as np

Array = np.ndarray


def _softmax_rows(z: Array) -> Array:
    """Row-wise softmax; entries equal to -inf get probability 0."""
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attn_fwd_intermediates(X: Array, Wqkv: Array, Wo: Array, S: int, H: int) -> Dict[str, Array]:
    """Q, K, V [B S, H dh], the attention output O [B S, H dh] and Y [B S, d]."""
    X = np.asarray(X, np.float64)
    Wqkv = np.asarray(Wqkv, np.float64)
    Wo = np.asarray(Wo, np.float64)
    M = X.shape[0]
    assert M % S == 0, "tokens must be whole sequences"
    dh = Wqkv.shape[1] // (3 * H)
    QKV = X @ Wqkv
    Q, K, V = QKV[:, :H * dh], QKV[:, H * dh:2 * H * dh], QKV[:, 2 * H * dh:]
    O = np.zeros_like(Q)
    future = np.triu(np.ones((S, S), dtype=bool), k=1)  # key index > query index
    for b in range(M // S):
        rows = slice(b * S, (b + 1) * S)
        for h in range(H):
            cols = slice(h * dh, (h + 1) * dh)
            scores = (Q[rows, cols] @ K[rows, cols].T) / math.sqrt(dh)
            scores[future] = -np.inf
            O[rows, cols] = _softmax_rows(scores) @ V[rows, cols]
    return {"Q": Q, "K": K, "V": V, "O": O, "Y": O @ Wo}


def attn_fwd(X: Array, Wqkv: Array, Wo: Array, S: int, H: int) -> Array:
    """Y of the causal multi-head self-attention block (unsharded)."""
    return attn_fwd_intermediates(X, Wqkv, Wo, S, H)["Y"]


def shard_qkv(Wqkv: Array, H: int, P: int, p: int) -> Array:
    """Columns of Wqkv that shard p owns: its heads' query, key and value columns, in that order."""
    dh = Wqkv.shape[1] // (3 * H)
    Hp = H // P
    blocks = [Wqkv[:, j * H * dh + p * Hp * dh: j * H * dh + (p + 1) * Hp * dh] for j in range(3)]
    return np.concatenate(blocks, axis=1)


def attn_fwd_sharded(X: Array, Wqkv: Array, Wo: Array, S: int, H: int, P: int, mu: int) -> Array:
    """The sliced block written out: mu chunks of whole sequences; per chunk and head
    shard p, the column-parallel projection of p's heads, their attention, the
    row-parallel partial O_p Wo_p; the P partials added in shard order."""
    X = np.asarray(X, np.float64)
    Wqkv = np.asarray(Wqkv, np.float64)
    Wo = np.asarray(Wo, np.float64)
    M = X.shape[0]
    B = M // S
    assert H % P == 0 and B % mu == 0
    dh = Wqkv.shape[1] // (3 * H)
    Hp = H // P
    rows_per_chunk = (B // mu) * S
    Y = np.zeros((M, Wo.shape[1]))
    for k in range(mu):
        rows = slice(k * rows_per_chunk, (k + 1) * rows_per_chunk)
        acc = np.zeros((rows_per_chunk, Wo.shape[1]))
        for p in range(P):
            Wo_p = Wo[p * Hp * dh:(p + 1) * Hp * dh]
            part = attn_fwd_intermediates(X[rows], shard_qkv(Wqkv, H, P, p), np.zeros((Hp * dh, 1)), S, Hp)
            acc = acc + part["O"] @ Wo_p
        Y[rows] = acc
    return Y
