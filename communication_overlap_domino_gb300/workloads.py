"""Workload shapes and seeded synthetic inputs for the sliced tensor-parallel MLP.

This module holds only shapes and random-number generation: none of the block's
arithmetic lives here, so that the fp64 oracle and the CUDA path can both draw
their inputs from it without sharing any of the computation.

Every tensor is produced in the plain mathematical layout of the block
``Y = act(X @ A) @ B``:

* ``X``  [M, d]         tokens x model width, ~N(0, 1)
* ``A``  [d, F]         column-parallel weight (GeLU / identity), ~N(0, 0.02)
* ``Wg``, ``Wu`` [d, F] gate and up weights (SwiGLU), ~N(0, 0.02)
* ``B``  [F, d]         row-parallel weight (``Wd`` for SwiGLU), ~N(0, 0.02)
* ``dY`` [M, d]         output gradient for the backward workloads, ~N(0, 1)

Tensor ``t`` (in the order X, A-or-(Wg, Wu), B, dY) is drawn from a CPU
``torch.Generator`` seeded with ``seed + t``, as fp32 ``randn`` times the
standard deviation, then rounded to bf16 (round-to-nearest-even).  The bf16
tensors are what the GPU receives; the oracle receives the same values widened
exactly to float64.

The shapes follow the tensor-parallel MLP of the Megatron-LM and LLaMA models
that the Domino page lists in "Builds on" (GPT-style GeLU MLP, Llama-style
SwiGLU MLP from "GLU Variants Improve Transformer").
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional, Tuple

import torch

WEIGHT_STD = 0.02
ACTS = ("gelu", "gelu_tanh", "swiglu", "identity")


@dataclass(frozen=True)
class Workload:
    """One sliced MLP problem: shapes, slicing factors and partial precision."""

    name: str
    M: int          # tokens (batch x sequence)
    d: int          # model width
    F: int          # hidden width (per gate/up projection for SwiGLU)
    P: int          # simulated tensor-parallel shards
    mu: int         # independent row chunks of X
    act: str        # "gelu" | "gelu_tanh" | "swiglu" | "identity"
    partial: str    # "f32" | "bf16": precision of each shard's partial output
    slices: int = 1  # column slices of the row-parallel output
    bwd: bool = False
    description: str = ""

    @property
    def Fp(self) -> int:
        return self.F // self.P

    @property
    def Mc(self) -> int:
        return self.M // self.mu

    def fwd_flops(self) -> int:
        """Algorithmic GEMM flops of one forward pass (2 per multiply-add)."""
        n_in = 2 if self.act == "swiglu" else 1
        return 2 * self.M * self.d * self.F * (n_in + 1)

    def bwd_flops(self) -> int:
        """Algorithmic GEMM flops of one backward pass (dX, dA, dB)."""
        return 2 * self.fwd_flops()

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("tiny_gelu_fwd", M=256, d=512, F=2048, P=2, mu=2, act="gelu", partial="f32",
                 description="Tiny GeLU MLP fwd: X[256 tokens (B=2,S=128), 512], A[512,2048], B[2048,512]; P=2, mu=2"),
        Workload("gpt_gelu_fwd", M=4096, d=2560, F=10240, P=4, mu=2, act="gelu", partial="f32",
                 description="GPT-style GeLU MLP fwd: X[4096 tokens (B=4,S=1024), 2560], A[2560,10240], B[10240,2560]; P=4, mu=2"),
        Workload("llama_swiglu_fwd", M=8192, d=4096, F=11008, P=8, mu=4, act="swiglu", partial="bf16",
                 description="Llama-style SwiGLU MLP fwd: X[8192,4096], gate/up[4096,11008], down[11008,4096]; P=8, mu=4"),
        Workload("llama_swiglu_fwdbwd", M=8192, d=4096, F=11008, P=8, mu=4, act="swiglu", partial="bf16", bwd=True,
                 description="Llama-style SwiGLU MLP fwd+bwd: shapes as llama_swiglu_fwd plus dY[8192,4096]; P=8, mu=4"),
        Workload("large_swiglu_fwd", M=16384, d=5120, F=13824, P=8, mu=4, act="swiglu", partial="bf16", slices=2,
                 description="Large SwiGLU MLP fwd: X[16384,5120], gate/up[5120,13824], down[13824,5120]; P=8, "
                             "mu in {1,2,4,8}, 2 output column slices"),
    )
}

# The workload the throughput benchmark times at one GPU: the largest configuration, at the mu (4) and the
# fused schedule that domino_mlp_plan picks for it on a GB300.
BENCH_WORKLOAD = "large_swiglu_fwd"


def _randn(shape: Tuple[int, ...], seed: int, std: float) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(torch.bfloat16)


def generate(w: Workload, seed: int = 0, with_dy: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Seeded bf16 CPU tensors for workload ``w`` in mathematical layout.

    Returns ``{"X", "A", "B"}`` (GeLU / identity) or ``{"X", "Wg", "Wu", "B"}``
    (SwiGLU; ``B`` is the down projection), plus ``"dY"`` when the workload has a
    backward pass or ``with_dy`` is true.
    """
    if with_dy is None:
        with_dy = w.bwd
    out: Dict[str, torch.Tensor] = {}
    t = 0
    out["X"] = _randn((w.M, w.d), seed + t, 1.0); t += 1
    if w.act == "swiglu":
        out["Wg"] = _randn((w.d, w.F), seed + t, WEIGHT_STD); t += 1
        out["Wu"] = _randn((w.d, w.F), seed + t, WEIGHT_STD); t += 1
    else:
        out["A"] = _randn((w.d, w.F), seed + t, WEIGHT_STD); t += 1
    out["B"] = _randn((w.F, w.d), seed + t, WEIGHT_STD); t += 1
    if with_dy:
        out["dY"] = _randn((w.M, w.d), seed + t, 1.0); t += 1
    return out


def to_float64(tensors: Dict[str, torch.Tensor]):
    """Exact widening of bf16 tensors to numpy float64 arrays (for the oracle)."""
    return {k: v.to(torch.float64).numpy() for k, v in tensors.items()}


# ----------------------------------------------------------- attention block

@dataclass(frozen=True)
class AttnWorkload:
    """One sliced attention problem: B sequences of S tokens, H heads of width dh."""

    name: str
    B: int          # sequences
    S: int          # tokens per sequence
    d: int          # model width
    H: int          # heads
    P: int          # simulated tensor-parallel shards (by heads)
    mu: int         # chunks of whole sequences
    partial: str    # "f32" | "bf16"
    dh: int = 128
    description: str = ""

    @property
    def M(self) -> int:
        return self.B * self.S

    def flops(self) -> int:
        """Algorithmic flops of one forward pass: the two projections and the causal attention core
        (Q K^T and P V over the S (S + 1) / 2 visible query-key pairs of each sequence and head)."""
        proj = 2 * self.M * self.d * 3 * self.H * self.dh + 2 * self.M * self.H * self.dh * self.d
        core = 2 * 2 * self.B * self.H * self.dh * (self.S * (self.S + 1) // 2)
        return proj + core

    def with_(self, **kw) -> "AttnWorkload":
        return replace(self, **kw)


ATTN_WORKLOADS: Dict[str, AttnWorkload] = {
    w.name: w
    for w in (
        AttnWorkload("tiny_attn_fwd", B=2, S=128, d=256, H=2, P=2, mu=2, partial="f32",
                     description="Tiny causal attention block: 2 sequences of 128 tokens, d=256, 2 heads; P=2, mu=2"),
        AttnWorkload("gpt_attn_fwd", B=4, S=1024, d=2560, H=20, P=4, mu=2, partial="f32",
                     description="Attention half of the GPT-style layer: 4 x 1024 tokens, d=2560, 20 heads of 128; "
                                 "P=4, mu=2"),
        AttnWorkload("llama_attn_fwd", B=4, S=2048, d=4096, H=32, P=8, mu=4, partial="bf16",
                     description="Attention half of the Llama-style layer: 4 x 2048 tokens, d=4096, 32 heads of 128; "
                                 "P=8, mu=4"),
    )
}


def generate_attn(w: AttnWorkload, seed: int = 0) -> Dict[str, torch.Tensor]:
    """Seeded bf16 CPU tensors in mathematical layout: ``X`` [B S, d] ~N(0, 1);
    ``Wqkv`` [d, 3 H dh] (all query heads, then key heads, then value heads) and
    ``Wo`` [H dh, d], ~N(0, 1/fan_in) so that projected entries have unit variance
    (for d = 2560 that is the 0.02 of the MLP weights).  Tensor t (X, Wqkv, Wo) is
    drawn with seed + t like ``generate``."""
    return {
        "X": _randn((w.M, w.d), seed, 1.0),
        "Wqkv": _randn((w.d, 3 * w.H * w.dh), seed + 1, w.d ** -0.5),
        "Wo": _randn((w.H * w.dh, w.d), seed + 2, (w.H * w.dh) ** -0.5),
    }

