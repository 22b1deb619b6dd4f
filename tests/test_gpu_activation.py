"""The fused activation epilogue, element by element (GB300, through the C ABI).

With one-hot rows of X (row i selects row i of A), every pre-activation is
exactly a chosen bf16 weight value, so the H the forward pass saves for the
backward is act(value) computed by the kernel's epilogue and rounded to bf16.
It is compared with the exact activation (the fp64 oracle's) rounded to bf16:
at most one bf16 unit in the last place apart, plus an absolute allowance of
1e-6 (1 + |x|) where the activation is tiny: fp32 cancellation in 1 + erf(z),
and the kernel's erf (Abramowitz & Stegun 7.1.26, absolute error <= 1.5e-7),
contribute up to ~|x| 1e-7 there (x Phi(x) at x = -8 is -5e-15).  The
pre-activation values cover [-8, 8] densely.
"""
import numpy as np
import pytest
import torch

import oracle
from communication_overlap_domino_gb300 import binding as b

pytestmark = pytest.mark.gpu

M, D, F, P = 512, 512, 2048, 2
FP = F // P


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _grid(lo, hi, seed, F=F):
    """d x F bf16 values covering [lo, hi], in a seeded order."""
    v = np.linspace(lo, hi, D * F)
    np.random.default_rng(seed).shuffle(v)
    return torch.tensor(v.reshape(D, F), dtype=torch.float32).to(torch.bfloat16)


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


@pytest.mark.parametrize("schedule", ["fused", "streams"])
@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "swiglu", "identity"])
def test_activation_epilogue_elementwise(act, schedule):
    _check_elementwise(act, schedule, F)


@pytest.mark.parametrize("schedule", ["fused", "streams"])
def test_swiglu_ragged_column_block_elementwise(schedule):
    # F / P = 1000 = 7 x 128 + 104: the last SwiGLU column block holds 104 valid columns of gate and of up (the
    # rest of its gate and up boxes zero-filled), and every one of them must pair gate column c with up column c
    _check_elementwise("swiglu", schedule, 2000)


def _check_elementwise(act, schedule, F):
    FP = F // P
    dev = torch.device("cuda:0")
    X = torch.zeros(M, D, dtype=torch.bfloat16)
    X[torch.arange(M), torch.arange(M) % D] = 1.0
    Wg = _grid(-8.0, 8.0, 1, F)
    Wu = _grid(-2.0, 2.0, 2, F)
    Bw = (0.02 * torch.randn(F, D, generator=torch.Generator().manual_seed(3))).to(torch.bfloat16)
    A = (Wg.to(dev), Wu.to(dev)) if act == "swiglu" else Wg.to(dev)
    A_sh, B_sh = b.shard_weights(A, Bw.to(dev), P)
    desc = b.make_desc(M, D, F, P, 2, act, "f32")
    saved = torch.zeros(b.saved_size(desc), dtype=torch.uint8, device=dev)
    b.mlp_fwd(X.to(dev), A_sh, B_sh, F=F, mu=2, act=act, partial="f32", schedule=schedule, saved=saved)
    torch.cuda.synchronize()

    nact = 2 if act == "swiglu" else 1
    shard_bytes = M * FP * (nact + 1) * 2
    raw = saved.cpu()
    H = torch.cat([raw[p * shard_bytes + M * nact * FP * 2:(p + 1) * shard_bytes].view(torch.bfloat16).view(M, FP)
                   for p in range(P)], dim=1).double().numpy()

    rows = np.arange(M) % D
    g = Wg.double().numpy()[rows]
    if act == "swiglu":
        exact = oracle.silu(g) * Wu.double().numpy()[rows]
    elif act == "gelu":
        exact = oracle.gelu(g)
    elif act == "gelu_tanh":
        exact = oracle.gelu_tanh(g)
    else:
        exact = g
    ref = torch.tensor(exact).to(torch.float32).to(torch.bfloat16).double().numpy()
    allow = _bf16_ulp(ref) + 1e-6 * (1.0 + np.abs(g))
    bad = np.abs(H - ref) > allow
    assert not bad.any(), (f"{act}/{schedule}: {int(bad.sum())} of {bad.size} elements off by more than one bf16 ulp; "
                           f"worst at x = {g[bad][0]}: got {H[bad][0]}, want {ref[bad][0]}")
