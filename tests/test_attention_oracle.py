"""The fp64 attention oracle against its pins, and planted mistakes the pins must catch (CPU only)."""
import math

import numpy as np
import pytest

import oracle.attention as att
from tests import attention_pins as pins

_good_inter = att.attn_fwd_intermediates
_good_sharded = att.attn_fwd_sharded
_good_shard_qkv = att.shard_qkv


@pytest.mark.parametrize("pin", pins.ALL_ATTN_PINS, ids=lambda f: f.__name__)
def test_attention_oracle_pin(pin):
    pin(att)


def _variant(scale_fn=None, mask=True, transpose=False, value_head_shift=0, softmax_axis=-1):
    """attn_fwd_intermediates with one step changed."""
    def inter(X, Wqkv, Wo, S, H):
        X = np.asarray(X, np.float64)
        Wqkv = np.asarray(Wqkv, np.float64)
        Wo = np.asarray(Wo, np.float64)
        dh = Wqkv.shape[1] // (3 * H)
        QKV = X @ Wqkv
        Q, K, V = QKV[:, :H * dh], QKV[:, H * dh:2 * H * dh], QKV[:, 2 * H * dh:]
        O = np.zeros_like(Q)
        future = np.triu(np.ones((S, S), dtype=bool), k=1)
        for b in range(X.shape[0] // S):
            rows = slice(b * S, (b + 1) * S)
            for h in range(H):
                c = slice(h * dh, (h + 1) * dh)
                hv = (h + value_head_shift) % H
                cv = slice(hv * dh, (hv + 1) * dh)
                z = (K[rows, c] @ Q[rows, c].T) if transpose else (Q[rows, c] @ K[rows, c].T)
                z = z * (scale_fn(dh) if scale_fn else 1.0 / math.sqrt(dh))
                if mask:
                    z[future] = -np.inf
                m = np.max(z, axis=softmax_axis, keepdims=True)
                e = np.exp(z - m)
                O[rows, c] = (e / np.sum(e, axis=softmax_axis, keepdims=True)) @ V[rows, cv]
        return {"Q": Q, "K": K, "V": V, "O": O, "Y": O @ Wo}
    return inter


def _sharded_drops_last(X, Wqkv, Wo, S, H, P, mu):
    Y = _good_sharded(X, Wqkv, Wo, S, H, P, mu)
    if P == 1:
        return Y
    dh = np.asarray(Wqkv).shape[1] // (3 * H)
    Hp = H // P
    part = att.attn_fwd_intermediates(X, _good_shard_qkv(Wqkv, H, P, P - 1), np.zeros((Hp * dh, 1)), S, Hp)["O"]
    return Y - part @ np.asarray(Wo)[(P - 1) * Hp * dh:]


def _shard_qkv_keys_of_next_shard(Wqkv, H, P, p):
    good = _good_shard_qkv(Wqkv, H, P, p)
    if P == 1:
        return good
    other = _good_shard_qkv(Wqkv, H, P, (p + 1) % P)
    w = good.shape[1] // 3
    return np.concatenate([good[:, :w], other[:, w:2 * w], good[:, 2 * w:]], axis=1)


MUTATIONS = {
    "no_causal_mask": ("attn_fwd_intermediates", _variant(mask=False)),
    "scale_one_over_dh": ("attn_fwd_intermediates", _variant(scale_fn=lambda dh: 1.0 / dh)),
    "no_scale": ("attn_fwd_intermediates", _variant(scale_fn=lambda dh: 1.0)),
    "scores_transposed": ("attn_fwd_intermediates", _variant(transpose=True)),
    "values_of_wrong_head": ("attn_fwd_intermediates", _variant(value_head_shift=1)),
    "softmax_over_queries": ("attn_fwd_intermediates", _variant(softmax_axis=0)),
    "sharded_drops_last_shard": ("attn_fwd_sharded", _sharded_drops_last),
    "shard_takes_next_shards_keys": ("shard_qkv", _shard_qkv_keys_of_next_shard),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_attention_pins_catch_mutation(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(att, attr, bad)
    failures = []
    for pin in pins.ALL_ATTN_PINS:
        try:
            pin(att)
        except (AssertionError, ValueError, FloatingPointError) as e:  # noqa: PERF203
            failures.append(f"{pin.__name__}: {e}")
    assert failures, f"mutation {name} passed every pin"
