"""Seeded synthetic inputs for causal attention workloads.

This module only draws random numbers; it holds none of the attention
arithmetic. The tests, the benchmark and the oracle checks all take their Q, K,
V and dO from here, so the CUDA path and the oracle see identical values.

Recipe (the pages print no workload data; this is the stated reading):
``torch.Generator('cpu').manual_seed(seed)``, then fp32 draws in the order
Q [B,T,Hq,Dh], K [B,T,Hkv,Dh], V [B,T,Hkv,Dh], dO [B,T,Hq,Dh]; each draw is
``randn`` unless the workload says uniform (``rand * 2 - 1``); the per-tensor
multiplier is applied in fp32; the result is then cast to the storage dtype.
The storage layout is the contiguous row-major [B,T,H,Dh] head split of [B,T,D]
activations from the "Architecture" page, "Tensor conventions".
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    Dh: int
    dtype: str  # "fp32" (TF32 MMA mode) or "bf16"
    seed: int
    mult: dict = field(default_factory=lambda: {"q": 1.0, "k": 1.0, "v": 1.0, "do": 1.0})
    uniform: tuple = ()  # names drawn as U(-1, 1) instead of N(0, 1)

    def __post_init__(self):
        for n in ("B", "Hq", "Hkv", "T", "Dh"):
            if getattr(self, n) < 1:
                raise ValueError(f"{n} must be >= 1")
        if self.Hq % self.Hkv:
            raise ValueError("Hq % Hkv must be 0")
        if self.dtype not in ("fp32", "bf16"):
            raise ValueError("dtype must be fp32 or bf16")

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def describe(self) -> str:
        h = f"H{self.Hq}" if self.Hq == self.Hkv else f"Hq{self.Hq} Hkv{self.Hkv}"
        return f"B{self.B} {h} T{self.T} Dh{self.Dh} {self.dtype}"


# The five workloads the attention path is specified on.
TINY = Workload("tiny_mha_tf32", 2, 4, 4, 64, 16, "fp32", 0)
GPT2S = Workload("gpt2s_mha_tf32", 8, 12, 12, 1024, 64, "fp32", 1,
                 mult={"q": 0.5, "k": 0.5, "v": 0.5, "do": 1.0})
HEADLINE = Workload("headline_mha_bf16", 4, 16, 16, 2048, 64, "bf16", 2)
GQA_LONG = Workload("gqa_long_bf16", 1, 32, 8, 8192, 128, "bf16", 3)
SKEWED = Workload("skewed_mha_bf16", 2, 8, 8, 4096, 128, "bf16", 4,
                  mult={"q": 3.0, "k": 3.0, "v": 1.0, "do": 1.0}, uniform=("v",))

WORKLOADS = (TINY, GPT2S, HEADLINE, GQA_LONG, SKEWED)
BY_NAME = {w.name: w for w in WORKLOADS}


def make_inputs(w: Workload, dtype: torch.dtype | None = None):
    """Return CPU tensors (q, k, v, do) in storage dtype, contiguous [B,T,H,Dh]."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    shapes = {
        "q": (w.B, w.T, w.Hq, w.Dh),
        "k": (w.B, w.T, w.Hkv, w.Dh),
        "v": (w.B, w.T, w.Hkv, w.Dh),
        "do": (w.B, w.T, w.Hq, w.Dh),
    }
    out = []
    for name in ("q", "k", "v", "do"):
        if name in w.uniform:
            x = torch.rand(shapes[name], generator=gen, dtype=torch.float32) * 2.0 - 1.0
        else:
            x = torch.randn(shapes[name], generator=gen, dtype=torch.float32)
        m = w.mult.get(name, 1.0)
        if m != 1.0:
            x = x * m
        out.append(x.to(dtype or w.torch_dtype).contiguous())
    return tuple(out)


def small(name: str, B, Hq, Hkv, T, Dh, dtype="bf16", seed=0, **kw) -> Workload:
    """An ad-hoc workload for edge-case tests (same recipe, other sizes)."""
    return Workload(name, B, Hq, Hkv, T, Dh, dtype, seed, **kw)
