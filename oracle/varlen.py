"""fp64 CPU oracle for causal attention over padded, variable-length rows.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` use it. It shares
no code with the CUDA path.

What it computes, and where the pages say so
--------------------------------------------
algo-v1-codepoint "docs/ARCHITECTURE.md", section "model.py": rows where no
key is allowed (fully padded) would make the softmax produce NaN, so they are
zeroed and masked again after it; masked scores must not let a NaN spread.
Neural-network page, "Stable softmax and cross-entropy": a fully masked slice
has no softmax (the full-sequence path rejects it).

Readings (the pages leave the layout open): a batch of B sequences padded on
the right to T positions, sequence b holding positions 0 .. L_b - 1 (0 <= L_b
<= T). Position t of sequence b is a padding position when t >= L_b; a padding
position is neither a query nor a key. So a real query attends causally to
the real keys before it (exactly the full-sequence oracle on the first L_b
positions), and every output at a padding position is zero: O, dQ, dK and dV
rows, and LSE is -inf there (the log of an empty sum). L_b = 0 is a sequence of
padding only, all of whose rows are fully masked: all zeros, no NaN. Gradients
flow only from real positions (the upstream gradient at padding positions is
ignored).

Parity status: pinned (see tests/test_oracle_varlen_pins.py): L_b = T is the
full-sequence oracle; changing anything at padding positions (inputs or the
upstream gradient) changes no output at a real position; padding outputs are
exactly zero; central finite differences of <dO, O> over the real positions.
"""

from __future__ import annotations

import numpy as np

from .attention import _check_shapes, attention_backward, attention_forward


def _lens(lens, b, t):
    lens = np.asarray(lens, dtype=np.int64)
    if lens.shape != (b,) or lens.min() < 0 or lens.max() > t:
        raise ValueError("lens must be B integers in [0, T]")
    return lens


def attention_forward_varlen(q, k, v, lens, scale: float | None = None):
    """Returns (O [B,T,Hq,Dh], LSE [B,Hq,T]) in fp64; zeros / -inf at padding."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    lens = _lens(lens, b, t)
    o = np.zeros((b, t, hq, dh))
    lse = np.full((b, hq, t), -np.inf)
    for bi in range(b):
        n = int(lens[bi])
        if n == 0:
            continue
        ob, lb = attention_forward(q[bi:bi + 1, :n], k[bi:bi + 1, :n], v[bi:bi + 1, :n], scale)
        o[bi, :n] = ob[0]
        lse[bi, :, :n] = lb[0]
    return o, lse


def attention_backward_varlen(q, k, v, do, lens, scale: float | None = None):
    """Returns (dQ, dK, dV) in fp64; zero rows at padding positions."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    lens = _lens(lens, b, t)
    dq = np.zeros((b, t, hq, dh))
    dk = np.zeros((b, t, hkv, dh))
    dv = np.zeros((b, t, hkv, dh))
    for bi in range(b):
        n = int(lens[bi])
        if n == 0:
            continue
        gq, gk, gv = attention_backward(q[bi:bi + 1, :n], k[bi:bi + 1, :n], v[bi:bi + 1, :n], do[bi:bi + 1, :n], scale)
        dq[bi, :n], dk[bi, :n], dv[bi, :n] = gq[0], gk[0], gv[0]
    return dq, dk, dv
