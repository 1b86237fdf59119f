"""fp64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
leg and ``--impl reference`` arm) use it. It shares no code with the CUDA path.

What it computes, and where the pages say so
--------------------------------------------
"Execution Backends and the Python ABI" (docs/internals/backends_and_python.html),
section "Incremental attention": the decoder issues one attention operation
per layer and token; query and output are [1, H, 1, d_h], viewed as [H, d_h];
the key and value pools are [physical_page, H, page_offset, d_h]; a
request-local table maps each logical page to a physical page ID of fixed
width; the CPU reference loops over the logical sequence and resolves each
K/V address through that table; the operation has no backward rule.

Readings taken where the pages are silent (also listed in the design notes):
the operation is batched over B requests, each with its own page table row
and cached length L_b (the pages' operation is B = 1); the new token attends
to every cached position 0 .. L_b - 1, its own key and value included (they
are appended to the cache before the operation); the scale is 1/sqrt(d_h);
with grouped-query pools (Hkv < Hq) query head h reads KV head floor(h / g),
g = Hq / Hkv, as in the full-sequence path (the pages' pools have one H:
Hkv = Hq is their case). The saved statistic is LSE = m + ln(l).

This is the plain definition written out: each key and value is fetched
through the page table position by position, the scores of the one query are
formed in fp64, and a max-subtracted softmax weights the values.

Parity status: pinned (see tests/test_oracle_paged_pins.py): equal to the last row
of the full-sequence causal oracle on a contiguous cache, invariant under a
permutation of the physical pages, the closed form for L = 1, and equal
outputs for equal queries of one group.
"""

from __future__ import annotations

import numpy as np

from .attention import contract, default_scale


def gather_positions(pool: np.ndarray, table_row: np.ndarray, length: int) -> np.ndarray:
    """[L, Hkv, Dh] = the first `length` logical positions of one request,
    each read from pool[table_row[t // page_size], :, t % page_size, :]."""
    page_size = pool.shape[2]
    rows = []
    for t in range(length):
        phys = int(table_row[t // page_size])
        rows.append(pool[phys, :, t % page_size, :])
    return np.stack(rows).astype(np.float64)


def kv_head(h: int, g: int) -> int:
    """KV head read by query head h when g query heads share one KV head
    (consecutive groups, as in the full-sequence path)."""
    return h // g


def paged_decode(q, k_pool, v_pool, page_table, seq_lens, scale: float | None = None):
    """q [B, Hq, Dh]; k_pool, v_pool [P, Hkv, page_size, Dh]; page_table
    [B, max_pages] (physical page IDs); seq_lens [B] (cached positions, >= 1).
    Returns (out [B, Hq, Dh], lse [B, Hq]) in fp64."""
    q = np.asarray(q, dtype=np.float64)
    k_pool = np.asarray(k_pool, dtype=np.float64)
    v_pool = np.asarray(v_pool, dtype=np.float64)
    B, Hq, Dh = q.shape
    Hkv = k_pool.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    if scale is None:
        scale = default_scale(Dh)
    out = np.zeros((B, Hq, Dh), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    for b in range(B):
        length = int(seq_lens[b])
        if length < 1:
            raise ValueError("every request needs at least one cached position")
        keys = gather_positions(k_pool, page_table[b], length)    # [L, Hkv, Dh]
        values = gather_positions(v_pool, page_table[b], length)  # [L, Hkv, Dh]
        for h in range(Hq):
            kv = kv_head(h, g)
            s = contract(keys[:, kv, :], q[b, h][:, None])[:, 0] * scale  # [L]
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            out[b, h] = contract((e / l)[None, :], values[:, kv, :])[0]
            lse[b, h] = m + np.log(l)
    return out, lse
