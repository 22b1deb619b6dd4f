"""Pins for the fp64 oracle: checks against something other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises ``AssertionError``
when the oracle disagrees with a fixed point of the mathematics:

* tabulated values of the normal CDF and of the logistic function (golden file);
* brute-force scalar loops (``math`` module, no numpy matmul, no scipy) on tiny
  inputs, so a transposed or mis-indexed operand shows up;
* central finite differences of the forward pass for every backward entry;
* the slicing invariants that the Domino page's Abstract rests on (the pieces are
  independent: the result does not depend on the number of row chunks, shards or
  column slices) and the Megatron-LM tensor-parallel identity (the sum over
  shards of the row-parallel partials is the unsharded product);
* closed forms: identity activation is associative, one-hot rows select a row of
  the weight, zero input gives zero output, hidden-unit permutations cancel.

They are plain functions (not tests) so that ``test_oracle_mutations`` can run
them against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "activation_table.txt")
ACTS = ("gelu", "gelu_tanh", "swiglu", "identity")


def load_activation_table():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(v) for v in line.split()])
    return np.array(rows)


def _rng(seed):
    return np.random.default_rng(seed)


def _weights(act, d, F, rng, scale=0.5):
    if act == "swiglu":
        return (rng.normal(0, scale, (d, F)), rng.normal(0, scale, (d, F)))
    return rng.normal(0, scale, (d, F))


def _close(a, b, rtol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    den = max(float(np.max(np.abs(b))), 1e-300)
    err = float(np.max(np.abs(a - b))) / den
    assert err <= rtol, f"{what}: relative error {err:.3e} > {rtol:.1e}"


# ---------------------------------------------------------------- activations

def pin_activation_table(orc):
    tab = load_activation_table()
    x, Phi, sig = tab[:, 0], tab[:, 1], tab[:, 2]
    _close(orc.gelu(x), x * Phi, 1e-14, "gelu vs x*Phi(x) table")
    _close(orc.sigmoid(x), sig, 1e-14, "sigmoid vs table")
    _close(orc.silu(x), x * sig, 1e-14, "silu vs x*sigma(x) table")
    # odd-part identities: f(x) - f(-x) = x for both x*Phi(x) and x*sigma(x)
    xs = np.linspace(-6, 6, 97)
    _close(orc.gelu(xs) - orc.gelu(-xs), xs, 1e-14, "gelu(x)-gelu(-x)=x")
    _close(orc.silu(xs) - orc.silu(-xs), xs, 1e-14, "silu(x)-silu(-x)=x")
    # the tanh form approximates the exact GeLU to a few 1e-4 and shares its limits
    assert float(np.max(np.abs(orc.gelu_tanh(xs) - orc.gelu(xs)))) < 1e-3, "gelu_tanh far from gelu"
    assert abs(float(orc.gelu_tanh(np.array([0.0]))[0])) == 0.0, "gelu_tanh(0) != 0"
    big = np.array([-12.0, 12.0])
    _close(orc.gelu_tanh(big), np.maximum(big, 0), 1e-12, "gelu_tanh tails")


def pin_activation_grads(orc):
    xs = np.linspace(-5, 5, 201)
    h = 1e-6
    for f, fp, name in ((orc.gelu, orc.gelu_grad, "gelu"), (orc.gelu_tanh, orc.gelu_tanh_grad, "gelu_tanh"),
                        (orc.silu, orc.silu_grad, "silu")):
        fd = (f(xs + h) - f(xs - h)) / (2 * h)
        _close(fp(xs), fd, 1e-8, f"{name}' vs central difference")
    # slopes at 0: both GeLU forms and SiLU have derivative 1/2 there
    for fp in (orc.gelu_grad, orc.gelu_tanh_grad, orc.silu_grad):
        assert abs(float(fp(np.array([0.0]))[0]) - 0.5) < 1e-15, "slope at 0 != 1/2"


# ------------------------------------------------------------ brute force fwd

def _scalar_act(act, g, u):
    if act == "gelu":
        return g * 0.5 * (1.0 + math.erf(g / math.sqrt(2.0)))
    if act == "gelu_tanh":
        return 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))
    if act == "swiglu":
        return g / (1.0 + math.exp(-g)) * u
    return g


def brute_force_fwd(X, A, B, act):
    """Scalar triple loops: Y[i][c] = sum_f act(sum_j X[i][j] A[j][f]) B[f][c]."""
    M, d = len(X), len(X[0])
    if act == "swiglu":
        Wg, Wu = A
        F = len(Wg[0])
    else:
        Wg, Wu = A, None
        F = len(A[0])
    dout = len(B[0])
    Y = [[0.0] * dout for _ in range(M)]
    for i in range(M):
        for f in range(F):
            g = 0.0
            u = 0.0
            for j in range(d):
                g += X[i][j] * Wg[j][f]
                if Wu is not None:
                    u += X[i][j] * Wu[j][f]
            h = _scalar_act(act, g, u)
            for c in range(dout):
                Y[i][c] += h * B[f][c]
    return np.array(Y)


def pin_brute_force_fwd(orc):
    rng = _rng(11)
    M, d, F = 3, 5, 7
    for act in ACTS:
        X = rng.normal(0, 1, (M, d))
        A = _weights(act, d, F, rng)
        B = rng.normal(0, 0.5, (F, d))
        ref = brute_force_fwd(X.tolist(), [a.tolist() for a in A] if act == "swiglu" else A.tolist(),
                              B.tolist(), act)
        _close(orc.mlp_fwd(X, A, B, act), ref, 1e-12, f"{act} fwd vs scalar loops")


# ------------------------------------------------------- finite-difference bwd

def _loss(orc, X, A, B, dY, act):
    return float(np.sum(orc.mlp_fwd(X, A, B, act) * dY))


def pin_fd_bwd(orc):
    """Every gradient entry against a central difference of <dY, Y> (4x8x16)."""
    rng = _rng(12)
    M, d, F = 4, 8, 16
    h = 1e-5
    for act in ACTS:
        X = rng.normal(0, 1, (M, d))
        A = _weights(act, d, F, rng)
        B = rng.normal(0, 0.5, (F, d))
        dY = rng.normal(0, 1, (M, d))
        g = orc.mlp_bwd(X, A, B, dY, act)
        params = {"dX": X, "dB": B}
        if act == "swiglu":
            params["dWg"], params["dWu"] = A[0], A[1]
        else:
            params["dA"] = A
        assert set(g) == set(params), f"{act}: gradient keys {sorted(g)}"
        for key, arr in params.items():
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                old = arr[idx]
                arr[idx] = old + h
                lp = _loss(orc, X, A, B, dY, act)
                arr[idx] = old - h
                lm = _loss(orc, X, A, B, dY, act)
                arr[idx] = old
                fd[idx] = (lp - lm) / (2 * h)
            _close(g[key], fd, 1e-7, f"{act} {key} vs finite differences")


# ------------------------------------------------------------------ invariants

def pin_sharded_equals_unsharded(orc):
    rng = _rng(13)
    M, d, F = 16, 8, 32
    for act in ACTS:
        X = rng.normal(0, 1, (M, d))
        A = _weights(act, d, F, rng)
        B = rng.normal(0, 0.5, (F, d))
        ref = orc.mlp_fwd(X, A, B, act)
        for P in (1, 2, 4, 8):
            for mu in (1, 2, 4):
                for S in (1, 2):
                    _close(orc.mlp_fwd_sharded(X, A, B, act, P, mu, S), ref, 1e-12,
                           f"{act} sharded P={P} mu={mu} S={S}")
        dY = rng.normal(0, 1, (M, d))
        gref = orc.mlp_bwd(X, A, B, dY, act)
        for P in (1, 2, 4):
            for mu in (1, 2, 4):
                gs = orc.mlp_bwd_sharded(X, A, B, dY, act, P, mu)
                for key in gref:
                    _close(gs[key], gref[key], 1e-12, f"{act} bwd sharded {key} P={P} mu={mu}")


def pin_row_separability(orc):
    rng = _rng(14)
    M, d, F = 12, 6, 10
    for act in ACTS:
        X = rng.normal(0, 1, (M, d))
        A = _weights(act, d, F, rng)
        B = rng.normal(0, 0.5, (F, d))
        Y = orc.mlp_fwd(X, A, B, act)
        rows = [0, 5, 11]
        _close(orc.mlp_fwd(X[rows], A, B, act), Y[rows], 1e-14, f"{act} rows")
        perm = rng.permutation(M)
        _close(orc.mlp_fwd(X[perm], A, B, act), Y[perm], 1e-14, f"{act} row permutation")
        dY = rng.normal(0, 1, (M, d))
        dX = orc.mlp_bwd(X, A, B, dY, act)["dX"]
        _close(orc.mlp_bwd(X[rows], A, B, dY[rows], act)["dX"], dX[rows], 1e-13, f"{act} dX rows")


def pin_hidden_permutation(orc):
    rng = _rng(15)
    M, d, F = 5, 6, 12
    for act in ACTS:
        X = rng.normal(0, 1, (M, d))
        A = _weights(act, d, F, rng)
        B = rng.normal(0, 0.5, (F, d))
        perm = rng.permutation(F)
        Ap = (A[0][:, perm], A[1][:, perm]) if act == "swiglu" else A[:, perm]
        _close(orc.mlp_fwd(X, Ap, B[perm], act), orc.mlp_fwd(X, A, B, act), 1e-13, f"{act} hidden permutation")


def pin_closed_forms(orc):
    rng = _rng(16)
    M, d, F = 6, 7, 9
    X = rng.normal(0, 1, (M, d))
    A = rng.normal(0, 0.5, (d, F))
    B = rng.normal(0, 0.5, (F, d))
    # identity activation: (X A) B == X (A B)
    _close(orc.mlp_fwd(X, A, B, "identity"), X @ (A @ B), 1e-13, "identity associativity")
    # one-hot rows select one row of A (and of Wg, Wu)
    c = 1.7
    for act in ACTS:
        W = _weights(act, d, F, rng)
        E = np.zeros((d, d))
        for j in range(d):
            E[j, j] = c
        Y = orc.mlp_fwd(E, W, B, act)
        for j in range(d):
            if act == "swiglu":
                hj = orc.silu(c * W[0][j]) * (c * W[1][j])
            elif act == "identity":
                hj = c * W[j]
            else:
                hj = getattr(orc, act)(c * W[j])
            _close(Y[j], hj @ B, 1e-13, f"{act} one-hot row {j}")
        # zero input gives zero output; Y is linear in B (and in Wu for SwiGLU)
        assert float(np.max(np.abs(orc.mlp_fwd(np.zeros((2, d)), W, B, act)))) == 0.0, f"{act} zero input"
        _close(orc.mlp_fwd(X, W, 3.0 * B, act), 3.0 * orc.mlp_fwd(X, W, B, act), 1e-13, f"{act} linear in B")
        if act == "swiglu":
            _close(orc.mlp_fwd(X, (W[0], -2.0 * W[1]), B, act), -2.0 * orc.mlp_fwd(X, W, B, act), 1e-13,
                   "swiglu linear in up")


def pin_shard_sum(orc):
    """The exchange step: one-hot partials, and the shard split of B (rows) summed
    over shards equals the unsharded row-parallel product."""
    rng = _rng(17)
    parts = [np.zeros((3, 4)) for _ in range(3)]
    for p in range(3):
        parts[p][p, p] = p + 1.0
    ref = np.zeros((3, 4))
    ref[0, 0], ref[1, 1], ref[2, 2] = 1.0, 2.0, 3.0
    _close(orc.shard_sum(parts), ref, 0.0, "shard_sum one-hot")
    H = rng.normal(0, 1, (5, 12))
    B = rng.normal(0, 1, (12, 6))
    for P in (1, 2, 3, 4):
        Fp = 12 // P
        parts = [H[:, p * Fp:(p + 1) * Fp] @ B[p * Fp:(p + 1) * Fp] for p in range(P)]
        _close(orc.shard_sum(parts), H @ B, 1e-13, f"shard_sum of row-parallel partials P={P}")


def pin_error_measure(orc):
    ref = np.array([[1.0, -4.0], [2.0, 0.5]])
    got = ref + np.array([[0.0, 0.02], [-0.04, 0.0]])
    assert abs(orc.max_rel_err(got, ref) - 0.01) < 1e-15, "max_rel_err"
    assert orc.max_rel_err(ref, ref) == 0.0


ALL_PINS = (
    pin_activation_table,
    pin_activation_grads,
    pin_brute_force_fwd,
    pin_fd_bwd,
    pin_sharded_equals_unsharded,
    pin_row_separability,
    pin_hidden_permutation,
    pin_closed_forms,
    pin_shard_sum,
    pin_error_measure,
)
