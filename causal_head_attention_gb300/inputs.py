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


# ---------------------------------------------------------------------------
# Paged decode (one new query token per request over a paged K/V cache)
# ---------------------------------------------------------------------------
#
# Recipe (the pages give the layout, not workload data; this is the stated
# reading): ``torch.Generator('cpu').manual_seed(seed)``, then in this order
#   lengths [B]  int, uniform in [1, max_len]; lengths[0] = max_len and, for
#                B >= 2, lengths[1] = 1 (the longest and the degenerate request);
#   q [B,Hq,Dh], k_pool, v_pool [P,Hkv,page_size,Dh]  randn (fp32, then cast);
#   a random permutation of the P physical pages, handed out to the requests in
#   order (request b takes ceil(L_b / page_size) pages); P is the pages needed
#   plus `spare` unused ones. Table entries past a request's last page are -1.
# Layout: "Execution Backends and the Python ABI", "Incremental attention":
# pools [physical_page, H, page_offset, d_h], a per-request table of physical
# page IDs, the query viewed as [H, d_h].


@dataclass(frozen=True)
class PagedWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Dh: int
    page_size: int
    max_len: int
    dtype: str  # "fp32" or "bf16"
    seed: int
    spare: int = 7

    def __post_init__(self):
        for n in ("B", "Hq", "Hkv", "Dh", "page_size", "max_len"):
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
    def max_pages(self) -> int:
        return -(-self.max_len // self.page_size)

    def describe(self) -> str:
        h = f"H{self.Hq}" if self.Hq == self.Hkv else f"Hq{self.Hq} Hkv{self.Hkv}"
        return f"B{self.B} {h} Dh{self.Dh} page{self.page_size} L<={self.max_len} {self.dtype}"


# Decode over the caches of the two model shapes the full-sequence path is
# specified on (16 heads of 64 up to 2048 positions; 32 query / 8 KV heads of
# 128 up to 8192 positions), plus small cases for the oracle.
DEC_SMALL = PagedWorkload("decode_small_gqa_bf16", 3, 4, 2, 64, 16, 300, "bf16", 10)
DEC_SMALL_F32 = PagedWorkload("decode_small_mha_fp32", 2, 4, 4, 32, 8, 100, "fp32", 11)
DEC_MHA = PagedWorkload("decode_mha_bf16", 64, 16, 16, 64, 16, 2048, "bf16", 12)
DEC_GQA = PagedWorkload("decode_gqa_bf16", 16, 32, 8, 128, 16, 8192, "bf16", 13)

PAGED_WORKLOADS = (DEC_SMALL, DEC_SMALL_F32, DEC_MHA, DEC_GQA)
PAGED_BY_NAME = {w.name: w for w in PAGED_WORKLOADS}


def make_paged_inputs(w: PagedWorkload, lengths=None):
    """Return CPU tensors (q, k_pool, v_pool, page_table int32, seq_lens int32).

    `lengths` (optional, B ints >= 1) replaces the drawn lengths; the rest of
    the recipe is unchanged."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    drawn = torch.randint(1, w.max_len + 1, (w.B,), generator=gen, dtype=torch.int64)
    drawn[0] = w.max_len
    if w.B >= 2:
        drawn[1] = 1
    if lengths is not None:
        drawn = torch.as_tensor(lengths, dtype=torch.int64).clone()
        if drawn.shape != (w.B,) or int(drawn.min()) < 1 or int(drawn.max()) > w.max_len:
            raise ValueError("lengths must be B ints in [1, max_len]")
    need = [-(-int(n) // w.page_size) for n in drawn]
    P = sum(need) + w.spare
    q = torch.randn((w.B, w.Hq, w.Dh), generator=gen, dtype=torch.float32)
    kp = torch.randn((P, w.Hkv, w.page_size, w.Dh), generator=gen, dtype=torch.float32)
    vp = torch.randn((P, w.Hkv, w.page_size, w.Dh), generator=gen, dtype=torch.float32)
    perm = torch.randperm(P, generator=gen)
    table = torch.full((w.B, w.max_pages), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    dt = w.torch_dtype
    return (q.to(dt).contiguous(), kp.to(dt).contiguous(), vp.to(dt).contiguous(), table,
            drawn.to(torch.int32))
