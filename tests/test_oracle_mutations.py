"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

Each mutation replaces one function of the oracle module with a wrong variant:
a dropped term, a wrong sign, a swapped or transposed operand, a missing shard,
a shifted chunk.  The pins of ``oracle_pins`` must reject every one of them.
"""
import numpy as np
import pytest

import oracle.oracle as orc
from tests import oracle_pins as pins

_good_inter = orc.mlp_fwd_intermediates
_good_bwd = orc.mlp_bwd
_good_sharded = orc.mlp_fwd_sharded
_good_bwd_sharded = orc.mlp_bwd_sharded


def _inter_swapped_gate_up(X, A, B, act):
    if act != "swiglu":
        return _good_inter(X, A, B, act)
    return _good_inter(X, (A[1], A[0]), B, act)


def _inter_transposed_B(X, A, B, act):
    r = _good_inter(X, A, B, act)
    B = np.asarray(B, np.float64)
    if B.shape[0] == B.shape[1]:
        r["Y"] = r["H"] @ B.T
    else:  # wrong rows of B when shapes allow only one product: reversed hidden order
        r["Y"] = r["H"] @ B[::-1]
    return r


def _bwd_drop_up_term(X, A, B, dY, act):
    out = _good_bwd(X, A, B, dY, act)
    if act == "swiglu":
        inter = orc.mlp_fwd_intermediates(X, A, B, act)
        dH = np.asarray(dY) @ np.asarray(B).T
        dg = dH * inter["u"] * orc.silu_grad(inter["g"])
        out["dX"] = dg @ np.asarray(A[0]).T
    return out


def _bwd_dB_from_preact(X, A, B, dY, act):
    out = _good_bwd(X, A, B, dY, act)
    inter = orc.mlp_fwd_intermediates(X, A, B, act)
    out["dB"] = inter["g"].T @ np.asarray(dY)
    return out


def _bwd_dA_transposed_input(X, A, B, dY, act):
    out = _good_bwd(X, A, B, dY, act)
    key = "dWg" if act == "swiglu" else "dA"
    out[key] = out[key] * 1.0 + 0.0
    out[key] = out[key][::-1]  # rows of X^T permuted: wrong index
    return out


def _sharded_drop_last(X, A, B, act, P, mu, slices=1):
    if P == 1:
        return _good_sharded(X, A, B, act, P, mu, slices)
    Y = _good_sharded(X, A, B, act, P, mu, slices)
    Fp = np.asarray(A[0] if act == "swiglu" else A).shape[1] // P
    last = slice((P - 1) * Fp, P * Fp)
    W = (np.asarray(A[0])[:, last], np.asarray(A[1])[:, last]) if act == "swiglu" else np.asarray(A)[:, last]
    return Y - orc.mlp_fwd(X, W, np.asarray(B)[last], act)


def _sharded_chunk_shift(X, A, B, act, P, mu, slices=1):
    Y = _good_sharded(X, A, B, act, P, mu, slices)
    if mu > 1:
        Mc = Y.shape[0] // mu
        Y = np.concatenate([Y[Mc:], Y[:Mc]])
    return Y


def _bwd_sharded_no_reduce(X, A, B, dY, act, P, mu):
    out = _good_bwd_sharded(X, A, B, dY, act, P, mu)
    out["dX"] = out["dX"] / P if P > 1 else out["dX"]
    return out


def _shard_sum_skips_first(partials):
    acc = np.zeros(np.asarray(partials[0]).shape)
    for z in partials[1:]:
        acc = acc + np.asarray(z, np.float64)
    return acc


MUTATIONS = {
    "shard_sum_skips_first_shard": ("shard_sum", _shard_sum_skips_first),
    "gelu_missing_half": ("gelu", lambda x: x * (1.0 + orc._erf(x / orc._SQRT2))),
    "gelu_wrong_scale": ("gelu", lambda x: 0.5 * x * (1.0 + orc._erf(x / 2.0))),
    "gelu_grad_missing_density": ("gelu_grad", lambda x: 0.5 * (1.0 + orc._erf(x / orc._SQRT2))),
    "gelu_tanh_wrong_sign": ("gelu_tanh", lambda x: 0.5 * x * (1.0 - np.tanh(orc._SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)))),
    "gelu_tanh_grad_missing_chain": ("gelu_tanh_grad", lambda x: 0.5 * (1.0 + np.tanh(orc._SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)))),
    "sigmoid_wrong_sign": ("sigmoid", lambda x: 1.0 / (1.0 + np.exp(x))),
    "silu_grad_missing_term": ("silu_grad", lambda x: orc.sigmoid(x)),
    "swiglu_gate_up_swapped": ("mlp_fwd_intermediates", _inter_swapped_gate_up),
    "row_parallel_weight_misindexed": ("mlp_fwd_intermediates", _inter_transposed_B),
    "bwd_dX_missing_up_term": ("mlp_bwd", _bwd_drop_up_term),
    "bwd_dB_uses_preactivation": ("mlp_bwd", _bwd_dB_from_preact),
    "bwd_dA_wrong_index": ("mlp_bwd", _bwd_dA_transposed_input),
    "sharded_drops_last_shard": ("mlp_fwd_sharded", _sharded_drop_last),
    "sharded_chunk_misplaced": ("mlp_fwd_sharded", _sharded_chunk_shift),
    "bwd_sharded_partials_not_summed": ("mlp_bwd_sharded", _bwd_sharded_no_reduce),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, bad)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:  # noqa: PERF203
            failures.append(f"{pin.__name__}: {e}")
    assert failures, f"mutation {name} passed every pin"
