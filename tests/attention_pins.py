"""Pins for the fp64 attention oracle: checks against something other than the oracle itself.

* brute-force scalar loops (``math`` module only) on tiny inputs: per query, the
  scaled dot products with the causally visible keys, their softmax and the
  weighted sum of values, then the output projection;
* closed forms: with all query weights zero every score is 0, so token t of a
  sequence averages the values of tokens 0..t (prefix means); one-token
  sequences make attention the identity, Y = X Wv Wo;
* causality (later tokens do not change earlier outputs, but do change later
  ones) and independence of sequences;
* head permutation (moving a head's query, key and value columns and its rows
  of Wo together) leaves Y unchanged;
* the slicing invariants: sequences in mu chunks and heads in P shards, with the
  row-parallel partials summed, equal the unsharded block.

Plain functions taking the oracle module, so ``test_attention_oracle`` can run
them against deliberately broken copies.
"""
from __future__ import annotations

import math

import numpy as np


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    den = max(float(np.max(np.abs(b))), 1e-300)
    err = float(np.max(np.abs(a - b))) / den
    assert err <= rtol, f"{what}: relative error {err:.3e} > {rtol:.1e}"


def _problem(seed, B, S, d, H, dh, scale=0.7):
    r = _rng(seed)
    return (r.normal(0, 1, (B * S, d)), r.normal(0, scale, (d, 3 * H * dh)), r.normal(0, scale, (H * dh, d)))


def brute_force_attn(X, Wqkv, Wo, S, H):
    M, d = len(X), len(X[0])
    dh = len(Wqkv[0]) // (3 * H)
    QKV = [[sum(X[i][c] * Wqkv[c][j] for c in range(d)) for j in range(3 * H * dh)] for i in range(M)]
    O = [[0.0] * (H * dh) for _ in range(M)]
    for i in range(M):
        b, t = divmod(i, S)
        for h in range(H):
            q = QKV[i][h * dh:(h + 1) * dh]
            scores = []
            for s in range(t + 1):
                k = QKV[b * S + s][H * dh + h * dh:H * dh + (h + 1) * dh]
                scores.append(sum(q[e] * k[e] for e in range(dh)) / math.sqrt(dh))
            top = max(scores)
            w = [math.exp(z - top) for z in scores]
            tot = sum(w)
            for e in range(dh):
                O[i][h * dh + e] = sum(w[s] / tot * QKV[b * S + s][2 * H * dh + h * dh + e] for s in range(t + 1))
    return [[sum(O[i][j] * Wo[j][c] for j in range(H * dh)) for c in range(d)] for i in range(M)]


def pin_attn_brute_force(att):
    for seed, (B, S, d, H, dh) in enumerate([(2, 3, 3, 2, 2), (1, 4, 2, 1, 3), (3, 2, 4, 3, 1)]):
        X, Wqkv, Wo = _problem(100 + seed, B, S, d, H, dh)
        want = brute_force_attn(X.tolist(), Wqkv.tolist(), Wo.tolist(), S, H)
        _close(att.attn_fwd(X, Wqkv, Wo, S, H), want, 1e-12, f"brute force B={B} S={S} H={H} dh={dh}")


def pin_attn_uniform_prefix_means(att):
    B, S, d, H, dh = 2, 5, 4, 2, 3
    X, Wqkv, Wo = _problem(7, B, S, d, H, dh)
    Wqkv[:, :H * dh] = 0.0  # all queries zero: every visible key scores 0
    V = X @ Wqkv[:, 2 * H * dh:]
    O = np.zeros_like(V)
    for b in range(B):
        run = np.zeros(H * dh)
        for t in range(S):
            run = run + V[b * S + t]
            O[b * S + t] = run / (t + 1)
    _close(att.attn_fwd(X, Wqkv, Wo, S, H), O @ Wo, 1e-12, "uniform attention = prefix means")


def pin_attn_single_token(att):
    B, d, H, dh = 6, 5, 2, 4
    X, Wqkv, Wo = _problem(8, B, 1, d, H, dh)
    _close(att.attn_fwd(X, Wqkv, Wo, 1, H), X @ Wqkv[:, 2 * H * dh:] @ Wo, 1e-12, "one-token sequences")


def pin_attn_causal_and_independent(att):
    B, S, d, H, dh = 3, 6, 4, 2, 2
    X, Wqkv, Wo = _problem(9, B, S, d, H, dh)
    Y = att.attn_fwd(X, Wqkv, Wo, S, H)
    t = 2
    X2 = X.copy()
    X2[S + t + 1:2 * S] += 1.0  # later tokens of sequence 1
    Y2 = att.attn_fwd(X2, Wqkv, Wo, S, H)
    _close(Y2[:S + t + 1], Y[:S + t + 1], 1e-13, "outputs up to token t do not see later tokens")
    _close(Y2[2 * S:], Y[2 * S:], 1e-13, "other sequences are independent")
    assert np.max(np.abs(Y2[S + t + 1:2 * S] - Y[S + t + 1:2 * S])) > 1e-6, "later outputs must change"
    X3 = X.copy()
    X3[S:S + t] += 1.0  # earlier tokens of sequence 1
    Y3 = att.attn_fwd(X3, Wqkv, Wo, S, H)
    assert np.max(np.abs(Y3[S + t] - Y[S + t])) > 1e-6, "token t must see earlier tokens"


def pin_attn_head_permutation(att):
    B, S, d, H, dh = 2, 4, 5, 3, 2
    X, Wqkv, Wo = _problem(10, B, S, d, H, dh)
    perm = [2, 0, 1]
    cols = [j * H * dh + h * dh + e for j in range(3) for h in perm for e in range(dh)]
    rows = [h * dh + e for h in perm for e in range(dh)]
    _close(att.attn_fwd(X, Wqkv[:, cols], Wo[rows], S, H), att.attn_fwd(X, Wqkv, Wo, S, H), 1e-12,
           "head permutation")


def pin_attn_sharded_equals_unsharded(att):
    B, S, d, H, dh = 4, 5, 6, 4, 3
    X, Wqkv, Wo = _problem(11, B, S, d, H, dh)
    ref = att.attn_fwd(X, Wqkv, Wo, S, H)
    for P in (1, 2, 4):
        for mu in (1, 2, 4):
            _close(att.attn_fwd_sharded(X, Wqkv, Wo, S, H, P, mu), ref, 1e-12, f"sharded P={P} mu={mu}")


ALL_ATTN_PINS = (
    pin_attn_brute_force,
    pin_attn_uniform_prefix_means,
    pin_attn_single_token,
    pin_attn_causal_and_independent,
    pin_attn_head_permutation,
    pin_attn_sharded_equals_unsharded,
)
