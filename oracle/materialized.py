"""fp64 CPU oracle for the materialized causal attention path and its
probability-returning diagnostic.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` use it. It shares
no code with the CUDA path.

What it computes, and where the pages say so
--------------------------------------------
"Execution Backends and the Python ABI" (docs/internals/backends_and_python.html),
section "What the Metal slice does": full-sequence attention has two exact
requests; the default materialized one returns probabilities and context and
keeps the [batch, heads, time, time] probabilities for its vector-Jacobian
products, and the explicit probability-returning diagnostic always takes that
path. Causal softmax there is one fused operation: scale, mask, normalise.

Because the probabilities are an output, the VJP takes an upstream gradient for
them as well as for the context. For the loss <dO, O> + <dP_up, P> of one head:

    dP = dO V^T + dP_up
    dS = P * (dP - rowsum(P * dP))        (the softmax VJP)
    dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO

With dP_up = 0 this is the full-sequence oracle's backward (there written with
D = rowsum(dO * O), which equals rowsum(P * dO V^T)). Readings: the
probabilities are float64 here and float32 on the device, [B, Hq, T, T], zero
above the diagonal; KV head floor(h / g) as in the full-sequence path.

The fused causal softmax itself (scale, mask, normalise) and its VJP with
respect to the unscaled scores are exposed as causal_softmax and
causal_softmax_vjp.

Parity status: pinned (see tests/test_oracle_materialized_pins.py): torch's fp64
softmax of the masked scores and its autograd, torch autograd through P and O,
central finite differences of the combined loss, the full-sequence oracle's
backward when dP_up = 0, and invariance to dP_up above the diagonal and to a
constant added to it on each row's kept entries.
"""

from __future__ import annotations

import numpy as np

from .attention import _check_shapes, contract, default_scale, head_forward


def causal_softmax(s, scale: float):
    """Fused causal softmax of [..., T, T] scores: P = softmax(scale * S) over
    j <= i (max subtracted), 0 above the diagonal; also LSE [..., T]."""
    s = np.asarray(s, dtype=np.float64) * scale
    t = s.shape[-1]
    keep = np.tril(np.ones((t, t), dtype=bool))
    s = np.where(keep, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=-1, keepdims=True)
    return e / l, (m + np.log(l))[..., 0]


def causal_softmax_vjp(p, g, scale: float):
    """Gradient of <G, causal_softmax(scale * S)> with respect to S."""
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    return scale * p * (g - np.sum(p * g, axis=-1, keepdims=True))


def attention_probs(q, k, v, scale: float | None = None):
    """Returns (O [B,T,Hq,Dh], P [B,Hq,T,T], LSE [B,Hq,T]) in fp64."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    scale = default_scale(dh) if scale is None else scale
    g = hq // hkv
    o = np.empty((b, t, hq, dh))
    p = np.empty((b, hq, t, t))
    lse = np.empty((b, hq, t))
    for bi in range(b):
        for h in range(hq):
            kv = h // g
            oh, lh, ph = head_forward(q[bi, :, h], k[bi, :, kv], v[bi, :, kv], scale)
            o[bi, :, h] = oh
            p[bi, h] = ph
            lse[bi, h] = lh
    return o, p, lse


def head_backward_probs(qh, kh, vh, doh, dph, p, scale: float):
    """VJP of one head of (O, P) with upstream (dO [T,Dh], dP_up [T,T] or None)."""
    qh, kh, vh, doh = (np.asarray(x, dtype=np.float64) for x in (qh, kh, vh, doh))
    dp = contract(doh, vh.T)
    if dph is not None:
        dp = dp + np.asarray(dph, dtype=np.float64)
    ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    return scale * contract(ds, kh), scale * contract(ds.T, qh), contract(p.T, doh)


def materialized_backward(q, k, v, do, dp=None, scale: float | None = None):
    """Whole tensors: (dQ, dK, dV) of <dO, O> + <dP, P>; dK, dV sum over each KV group."""
    b, t, hq, hkv, dh = _check_shapes(q, k, v)
    scale = default_scale(dh) if scale is None else scale
    g = hq // hkv
    dq = np.empty((b, t, hq, dh))
    dk = np.zeros((b, t, hkv, dh))
    dv = np.zeros((b, t, hkv, dh))
    for bi in range(b):
        for h in range(hq):
            kv = h // g
            qh, kh, vh = q[bi, :, h], k[bi, :, kv], v[bi, :, kv]
            _, _, ph = head_forward(qh, kh, vh, scale)
            dqh, dkh, dvh = head_backward_probs(qh, kh, vh, do[bi, :, h], None if dp is None else dp[bi, h], ph,
                                                scale)
            dq[bi, :, h] = dqh
            dk[bi, :, kv] += dkh
            dv[bi, :, kv] += dvh
    return dq, dk, dv
