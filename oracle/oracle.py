"""Oracle for the sliced tensor-parallel MLP block: plain, slow, fp64, CPU.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module; it
is used by the tests, by ``__graft_entry__.smoke()`` and by the benchmark's
CPU-baseline leg.  It shares no code with the CUDA path.

What it computes
----------------
The Domino page ("Domino: Eliminating Communication in LLM Training via Generic
Tensor Slicing and Overlapping", Abstract) states the method: the data
dependency of one batch is broken into smaller independent pieces whose
communication is overlapped with the computation of the next piece.  The
method changes the order of the work, not its result, so the oracle is the
plain *unsharded* transformer MLP block in float64:

* GeLU (GPT-style):   ``Y = gelu(X A) B``
* SwiGLU (Llama-style, "GLU Variants Improve Transformer", listed under
  "Builds on" on the Domino page):  ``Y = (silu(X Wg) * (X Wu)) Wd``

with the tensor-parallel split of the Megatron-LM MLP (also under "Builds on"):
A is split by columns and B by rows into P shards, and the sum over shards of
each shard's partial output equals the unsharded product.  The backward pass
is the chain rule of the same block.  ``mlp_fwd_sharded`` /
``mlp_bwd_sharded`` write the slicing out explicitly (row chunks, shards,
output column slices, partial sums added in shard order); they exist only so
that the tests can check the slicing invariants against the unsharded form.

Readings where the pages are silent (all recorded in the design notes):
GeLU is the exact erf form (a tanh form is a separate activation); there are
no biases; SwiGLU is ``silu(gate) * up``; the intermediate activation and the
partials are kept in fp64 here (the GPU rounds them, the tolerance absorbs it).

Pins: every function here is checked in ``tests/test_oracle.py`` against
brute-force scalar loops, closed forms, finite differences and the slicing
invariants; ``tests/test_oracle_mutations.py`` plants mistakes in this module
and checks that the pins catch them.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple, Union

import numpy as np
from scipy.special import erf as _erf

Array = np.ndarray
Weights = Union[Array, Tuple[Array, Array]]

_SQRT2 = math.sqrt(2.0)
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


# --------------------------------------------------------------------------
# Activations and their derivatives (fp64, elementwise)
# --------------------------------------------------------------------------

def sigmoid(x: Array) -> Array:
    """Logistic function 1 / (1 + exp(-x))."""
    return 1.0 / (1.0 + np.exp(-x))


def gelu(x: Array) -> Array:
    """Exact GeLU: x * Phi(x), Phi the standard normal CDF = (1 + erf(x/sqrt 2)) / 2."""
    return 0.5 * x * (1.0 + _erf(x / _SQRT2))


def gelu_grad(x: Array) -> Array:
    """d/dx [x Phi(x)] = Phi(x) + x phi(x), phi the standard normal density."""
    return 0.5 * (1.0 + _erf(x / _SQRT2)) + x * _INV_SQRT_2PI * np.exp(-0.5 * x * x)


def gelu_tanh(x: Array) -> Array:
    """tanh approximation of GeLU: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)))


def gelu_tanh_grad(x: Array) -> Array:
    """Derivative of ``gelu_tanh`` by the product and chain rules."""
    inner = _SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)
    t = np.tanh(inner)
    dinner = _SQRT_2_OVER_PI * (1.0 + 3.0 * 0.044715 * x * x)
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * dinner


def silu(x: Array) -> Array:
    """SiLU (swish with beta = 1): x * sigmoid(x)."""
    return x * sigmoid(x)


def silu_grad(x: Array) -> Array:
    """d/dx [x sigmoid(x)] = sigmoid(x) (1 + x (1 - sigmoid(x)))."""
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


_PLAIN_ACTS = {
    "gelu": (gelu, gelu_grad),
    "gelu_tanh": (gelu_tanh, gelu_tanh_grad),
    "identity": (lambda x: x, lambda x: np.ones_like(x)),
}


def _split(act: str, A: Weights):
    if act == "swiglu":
        Wg, Wu = A
        return np.asarray(Wg, np.float64), np.asarray(Wu, np.float64)
    if act not in _PLAIN_ACTS:
        raise ValueError(f"unknown activation {act!r}")
    return np.asarray(A, np.float64), None


# --------------------------------------------------------------------------
# The unsharded block
# --------------------------------------------------------------------------

def mlp_fwd_intermediates(X: Array, A: Weights, B: Array, act: str) -> Dict[str, Array]:
    """Forward pass keeping the pre-activations and the hidden activation.

    Returns ``g`` (= X A or X Wg), ``u`` (= X Wu, SwiGLU only), ``H`` (the
    activated hidden layer) and ``Y`` (= H B).
    """
    X = np.asarray(X, np.float64)
    B = np.asarray(B, np.float64)
    W0, W1 = _split(act, A)
    g = X @ W0
    if act == "swiglu":
        u = X @ W1
        H = silu(g) * u
    else:
        u = None
        H = _PLAIN_ACTS[act][0](g)
    Y = H @ B
    return {"g": g, "u": u, "H": H, "Y": Y}


def mlp_fwd(X: Array, A: Weights, B: Array, act: str) -> Array:
    """``Y = act(X A) B`` (SwiGLU: ``(silu(X Wg) * (X Wu)) Wd``) in float64."""
    return mlp_fwd_intermediates(X, A, B, act)["Y"]


def mlp_bwd(X: Array, A: Weights, B: Array, dY: Array, act: str) -> Dict[str, Array]:
    """Gradients of ``<dY, Y>`` with respect to X, A (or Wg, Wu) and B.

    Chain rule of the block, with g = X A (or X Wg), u = X Wu:

    * dH = dY B^T
    * plain act:  dG = dH * act'(g);  dX = dG A^T;  dA = X^T dG
    * SwiGLU:     dg = dH * u * silu'(g);  du = dH * silu(g);
                  dX = dg Wg^T + du Wu^T;  dWg = X^T dg;  dWu = X^T du
    * dB = H^T dY
    """
    X = np.asarray(X, np.float64)
    B = np.asarray(B, np.float64)
    dY = np.asarray(dY, np.float64)
    W0, W1 = _split(act, A)
    inter = mlp_fwd_intermediates(X, A, B, act)
    g, u, H = inter["g"], inter["u"], inter["H"]
    dH = dY @ B.T
    out: Dict[str, Array] = {"dB": H.T @ dY}
    if act == "swiglu":
        dg = dH * u * silu_grad(g)
        du = dH * silu(g)
        out["dX"] = dg @ W0.T + du @ W1.T
        out["dWg"] = X.T @ dg
        out["dWu"] = X.T @ du
    else:
        dG = dH * _PLAIN_ACTS[act][1](g)
        out["dX"] = dG @ W0.T
        out["dA"] = X.T @ dG
    return out


# --------------------------------------------------------------------------
# The sliced form, written out step by step (for the invariant tests)
# --------------------------------------------------------------------------

def _shard_cols(W: Array, P: int, p: int) -> Array:
    Fp = W.shape[1] // P
    return W[:, p * Fp:(p + 1) * Fp]


def mlp_fwd_sharded(X: Array, A: Weights, B: Array, act: str, P: int, mu: int, slices: int = 1) -> Array:
    """Forward pass computed piece by piece, as the sliced schedule orders it.

    X is split into ``mu`` row chunks; A (or Wg and Wu) into ``P`` column
    shards; B into the matching ``P`` row shards; the output columns into
    ``slices`` slices.  For each chunk k and slice s, shard p produces the
    partial ``Z[k,p,s] = act(X_k A_p) B_p[:, s]``; the partials are summed in
    shard order p = 0..P-1 (the stand-in for the tensor-parallel all-reduce)
    to give ``Y_k[:, s]``.
    """
    X = np.asarray(X, np.float64)
    B = np.asarray(B, np.float64)
    M, d = X.shape
    W0, W1 = _split(act, A)
    F = W0.shape[1]
    if M % mu or F % P or d % slices:
        raise ValueError("mu must divide M, P must divide F and slices must divide d")
    Mc, Fp, ds = M // mu, F // P, d // slices
    Y = np.zeros((M, d))
    for k in range(mu):
        Xk = X[k * Mc:(k + 1) * Mc]
        for s in range(slices):
            acc = np.zeros((Mc, ds))
            for p in range(P):
                g = Xk @ _shard_cols(W0, P, p)
                if act == "swiglu":
                    H = silu(g) * (Xk @ _shard_cols(W1, P, p))
                else:
                    H = _PLAIN_ACTS[act][0](g)
                Bp = B[p * Fp:(p + 1) * Fp, s * ds:(s + 1) * ds]
                acc = acc + H @ Bp
            Y[k * Mc:(k + 1) * Mc, s * ds:(s + 1) * ds] = acc
    return Y


def mlp_bwd_sharded(X: Array, A: Weights, B: Array, dY: Array, act: str, P: int, mu: int) -> Dict[str, Array]:
    """Backward pass piece by piece: per chunk k and shard p, the shard's
    partial input gradient is formed and the partials are summed over p (the
    all-reduce of dX); the weight gradients of shard p are accumulated over
    the chunks and placed in shard p's columns (rows, for B)."""
    X = np.asarray(X, np.float64)
    B = np.asarray(B, np.float64)
    dY = np.asarray(dY, np.float64)
    M, d = X.shape
    W0, W1 = _split(act, A)
    F = W0.shape[1]
    if M % mu or F % P:
        raise ValueError("mu must divide M and P must divide F")
    Mc, Fp = M // mu, F // P
    dX = np.zeros((M, d))
    dW0 = np.zeros_like(W0)
    dW1 = np.zeros_like(W0) if act == "swiglu" else None
    dB = np.zeros_like(B)
    for k in range(mu):
        rows = slice(k * Mc, (k + 1) * Mc)
        Xk, dYk = X[rows], dY[rows]
        acc = np.zeros((Mc, d))
        for p in range(P):
            cols = slice(p * Fp, (p + 1) * Fp)
            W0p = W0[:, cols]
            Bp = B[cols, :]
            g = Xk @ W0p
            dH = dYk @ Bp.T
            if act == "swiglu":
                W1p = W1[:, cols]
                u = Xk @ W1p
                H = silu(g) * u
                dg = dH * u * silu_grad(g)
                du = dH * silu(g)
                acc = acc + (dg @ W0p.T + du @ W1p.T)
                dW0[:, cols] += Xk.T @ dg
                dW1[:, cols] += Xk.T @ du
            else:
                H = _PLAIN_ACTS[act][0](g)
                dG = dH * _PLAIN_ACTS[act][1](g)
                acc = acc + dG @ W0p.T
                dW0[:, cols] += Xk.T @ dG
            dB[cols, :] += H.T @ dYk
        dX[rows] = acc
    out = {"dX": dX, "dB": dB}
    if act == "swiglu":
        out["dWg"], out["dWu"] = dW0, dW1
    else:
        out["dA"] = dW0
    return out


def max_rel_err(got, ref) -> float:
    """max|got - ref| / max|ref|: the error measure the parity tests use."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def shard_sum(partials) -> Array:
    """The exchange step alone: Y = sum over shards of the partial outputs, in fp64.

    Stands in for the tensor-parallel all-reduce of the row-parallel products
    (Megatron-LM MLP; hidden by Domino behind the next piece's computation,
    Domino page, Abstract).
    """
    acc = np.zeros(np.asarray(partials[0]).shape)
    for z in partials:
        acc = acc + np.asarray(z, np.float64)
    return acc
