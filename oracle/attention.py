"""fp64 CPU oracle for causal multi-head self-attention: forward and its VJP.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline
leg and ``--impl reference`` arm) use it. It shares no code with the CUDA path.

What it computes, and where the pages say so
--------------------------------------------
Sources are the riftco-transformer documentation pages:

* "Architecture" (docs/concepts/architecture.html), section "Tensor
  conventions": storage is contiguous row-major, activations are [B,T,D], attention
  scores are laid out [B,H,T_q,T_k], and a key at position t_k is not used by a
  query at t_q when t_k > t_q.
* Neural-network page (docs/learn/neural_network.html), section "Stable
  softmax and cross-entropy": softmax subtracts the row maximum before
  exponentiating and allows -inf entries from the causal mask; section "Where
  attention is": scaled causal attention over split heads.
* "Execution Backends and the Python ABI" (docs/internals/backends_and_python.html),
  section "What the Metal slice does": the materialized path and the Flash path
  are both exact; Flash keeps only per-row [B,H,T] statistics and its backward
  recomputes scores and probabilities from Q, K and those statistics.
* algo-v1-codepoint "docs/ARCHITECTURE.md", section "config.py": grouped-query
  attention needs num_query_heads % num_kv_heads == 0.

Readings taken where the pages are silent (also listed in the design notes):
the scale is 1/sqrt(Dh); the diagonal key (t_k == t_q) is kept; query head h
reads KV head floor(h / g) with g = Hq / Hkv; the saved row statistic is
LSE = m + ln(l) (natural log), equivalent to the pages' separate max and sum.

This is the plain definition written out: the full T x T score matrix of each
head is materialised in fp64, masked, normalised with a max-subtracted softmax,
and multiplied by V. The backward is the textbook softmax VJP on that
materialised matrix. There is no tiling, fusion or reordering.

Parity status: pinned (see tests/test_oracle_pins.py): row sums, closed forms
for T=1 and Q=0, causality, key-shift invariance, the large-logit example,
the D identity, central finite differences, an independent online-softmax
(tile-8) recomputation, torch's fp64 scaled_dot_product_attention, and the
pages' worked matmul example for the contraction helper.

Layouts: q, dO: [B, T, Hq, Dh]; k, v: [B, T, Hkv, Dh]; LSE: [B, Hq, T].
All outputs are float64 numpy arrays.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "contract",
    "default_scale",
    "head_forward",
    "head_backward",
    "attention_forward",
    "attention_backward",
    "group_reference",
]


def contract(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Plain fp64 matrix product a @ b (the one contraction every step uses).

    Pinned by the worked example on "Execution Backends and the Python ABI",
    section "Python client": [[1,2,3],[4,5,6]] @ [[7,8],[9,10],[11,12]]
    = [[58,64],[139,154]].
    """
    return np.matmul(np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64))


def default_scale(dh: int) -> float:
    """1/sqrt(Dh): the reading taken for the pages' unstated score scale."""
    return 1.0 / math.sqrt(dh)


def _causal_keep(t: int) -> np.ndarray:
    """keep[i, j] is True when key j may be used by query i, i.e. j <= i.

    "Architecture" page, "Tensor conventions": keys with t_k > t_q are dropped.
    """
    return np.tril(np.ones((t, t), dtype=bool))


def head_forward(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, scale: float):
    """One head. qh, kh, vh: [T, Dh]. Returns (O [T,Dh], LSE [T], P [T,T]).

    1. S = scale * Q K^T, the full [T, T] score matrix.
    2. Entries with j > i are excluded (set to -inf, so their probability is 0).
    3. Stable softmax per row: m = max_j S, e = exp(S - m), l = sum_j e,
       P = e / l, LSE = m + ln(l).
    4. O = P V.
    """
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    t = qh.shape[0]
    if t < 1:
        raise ValueError("a fully masked (empty) softmax row is rejected")
    s = scale * contract(qh, kh.T)
    s = np.where(_causal_keep(t), s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)  # finite: key 0 is always kept
    e = np.exp(s - m)  # exp(-inf) == 0 exactly for masked entries
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    lse = (m + np.log(l))[:, 0]
    o = contract(p, vh)
    return o, lse, p


def head_backward(qh, kh, vh, oh, doh, p, scale: float):
    """VJP of one head given the forward's O and P (all [T, *] fp64).

    dV = P^T dO
    dP = dO V^T
    D_i = sum_d dO[i,d] O[i,d]          (equals sum_j P[i,j] dP[i,j])
    dS = P * (dP - D)                    (softmax VJP; masked entries stay 0)
    dQ = scale * dS K
    dK = scale * dS^T Q
    Returns (dQ, dK, dV, D).
    """
    qh = np.asarray(qh, dtype=np.float64)
    kh = np.asarray(kh, dtype=np.float64)
    vh = np.asarray(vh, dtype=np.float64)
    oh = np.asarray(oh, dtype=np.float64)
    doh = np.asarray(doh, dtype=np.float64)
    dv = contract(p.T, doh)
    dp = contract(doh, vh.T)
    d = np.sum(doh * oh, axis=1)
    ds = p * (dp - d[:, None])
    dq = scale * contract(ds, kh)
    dk = scale * contract(ds.T, qh)
    return dq, dk, dv, d


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, T, H, Dh]")
    b, t, hq, dh = q.shape
    if k.shape != v.shape or k.shape[0] != b or k.shape[1] != t or k.shape[3] != dh:
        raise ValueError("k and v must be [B, T, Hkv, Dh] matching q")
    hkv = k.shape[2]
    if hq % hkv != 0:
        raise ValueError("grouped-query attention needs Hq % Hkv == 0")
    return b, t, hq, hkv, dh


def attention_forward(q, k, v, scale: float | None = None):
    """Whole tensors. Returns (O [B,T,Hq,Dh], LSE [B,Hq,T]) in fp64."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    scale = default_scale(dh) if scale is None else scale
    g = hq // hkv
    o = np.empty((b, t, hq, dh), dtype=np.float64)
    lse = np.empty((b, hq, t), dtype=np.float64)
    for bi in range(b):
        for h in range(hq):
            kv = h // g
            oh, lh, _ = head_forward(q[bi, :, h], k[bi, :, kv], v[bi, :, kv], scale)
            o[bi, :, h] = oh
            lse[bi, h] = lh
    return o, lse


def attention_backward(q, k, v, do, scale: float | None = None, o=None):
    """Whole tensors. Returns (dQ, dK, dV) in fp64; dK/dV sum over each KV group.

    o: the forward output the backward is handed ([B,T,Hq,Dh]), from which
    D = rowsum(dO * O) is formed, as a backward that takes the stored output
    as an argument does. None: the oracle's own exact forward output, which
    gives the exact VJP (the two agree when o is that output)."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    scale = default_scale(dh) if scale is None else scale
    g = hq // hkv
    dq = np.empty((b, t, hq, dh), dtype=np.float64)
    dk = np.zeros((b, t, hkv, dh), dtype=np.float64)
    dv = np.zeros((b, t, hkv, dh), dtype=np.float64)
    for bi in range(b):
        for h in range(hq):
            kv = h // g
            qh, kh, vh = q[bi, :, h], k[bi, :, kv], v[bi, :, kv]
            oh, _, p = head_forward(qh, kh, vh, scale)
            if o is not None:
                oh = np.asarray(o[bi, :, h], dtype=np.float64)
            dqh, dkh, dvh, _ = head_backward(qh, kh, vh, oh, do[bi, :, h], p, scale)
            dq[bi, :, h] = dqh
            dk[bi, :, kv] += dkh
            dv[bi, :, kv] += dvh
    return dq, dk, dv


def group_reference(q, k, v, do, b: int, kv: int, scale: float | None = None, o=None):
    """Forward and backward for one (batch, KV head) group: its g query heads.

    This is how full-size workloads are checked on a sample: every output of the
    sampled group is computed exactly, element by element comparable.
    Returns a dict with O [T,g,Dh], LSE [g,T], D [g,T], dQ [T,g,Dh],
    dK [T,Dh], dV [T,Dh], all fp64. When o ([B,T,Hq,Dh], the output a backward
    is handed) is given, the dict also holds "given_o": the backward's dQ, dK,
    dV and D with D = rowsum(dO * o) instead of the exact output.
    """
    _, t, hq, hkv, dh = _check_shapes(q, k, v)
    scale = default_scale(dh) if scale is None else scale
    g = hq // hkv
    kh = np.asarray(k[b, :, kv], dtype=np.float64)
    vh = np.asarray(v[b, :, kv], dtype=np.float64)
    out = {
        "O": np.empty((t, g, dh)),
        "LSE": np.empty((g, t)),
        "D": np.empty((g, t)),
        "dQ": np.empty((t, g, dh)),
        "dK": np.zeros((t, dh)),
        "dV": np.zeros((t, dh)),
    }
    if o is not None:
        out["given_o"] = {"D": np.empty((g, t)), "dQ": np.empty((t, g, dh)), "dK": np.zeros((t, dh)),
                          "dV": np.zeros((t, dh))}
    for r in range(g):
        h = kv * g + r
        qh = np.asarray(q[b, :, h], dtype=np.float64)
        oh, lh, p = head_forward(qh, kh, vh, scale)
        dqh, dkh, dvh, d = head_backward(qh, kh, vh, oh, do[b, :, h], p, scale)
        out["O"][:, r] = oh
        out["LSE"][r] = lh
        out["D"][r] = d
        out["dQ"][:, r] = dqh
        out["dK"] += dkh
        out["dV"] += dvh
        if o is not None:
            go = out["given_o"]
            dqh, dkh, dvh, d = head_backward(qh, kh, vh, np.asarray(o[b, :, h], dtype=np.float64), do[b, :, h],
                                             p, scale)
            go["D"][r] = d
            go["dQ"][:, r] = dqh
            go["dK"] += dkh
            go["dV"] += dvh
    return out
