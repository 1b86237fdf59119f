"""Helpers shared by the parity tests: tolerances, error metric, oracle calls."""

from __future__ import annotations

import numpy as np

import oracle

# Relative Frobenius error bounds for the attention path, per storage dtype:
# bf16 operands with fp32 accumulation, or fp32 storage with TF32 operands.
TOL = {
    "bf16": {"O": 5e-3, "LSE": 1e-3, "dQ": 1e-2, "dK": 1e-2, "dV": 1e-2},
    "fp32": {"O": 1e-3, "LSE": 1e-3, "dQ": 3e-3, "dK": 3e-3, "dV": 3e-3},
}


def rel_fro(got, ref, den=None) -> float:
    """||got - ref||_F / ||ref||_F in fp64 (or / den when given)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if den is None:
        den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.linalg.norm(got - ref))
    return float(np.linalg.norm(got - ref) / den)


def uncancelled_norms(q, k, v, do):
    """For T = 1, dQ and dK vanish identically (dS = P (dP - D) with P = 1 and
    D = dP): their relative error is undefined. The error is then measured
    against the size of the terms that cancel, scale * (P * dP) K for dQ and
    scale * (P * dP)^T Q for dK. Returns (||.||_F for dQ, for dK)."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    assert q.shape[1] == 1
    g = q.shape[2] // k.shape[2]
    scale = oracle.default_scale(q.shape[3])
    kk = np.repeat(k, g, axis=2)
    vv = np.repeat(v, g, axis=2)
    dp = np.sum(do * vv, axis=-1, keepdims=True)  # [B,1,Hq,1]
    return float(np.linalg.norm(scale * dp * kk)), float(np.linalg.norm(scale * dp * q))


def to64(t) -> np.ndarray:
    """torch tensor (any device/dtype) -> fp64 numpy, exact upcast of the stored values."""
    return t.detach().to("cpu").double().numpy()


def full_reference(q, k, v, do):
    """Whole-tensor oracle outputs as a dict of fp64 arrays."""
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    o, lse = oracle.attention_forward(q64, k64, v64)
    dq, dk, dv = oracle.attention_backward(q64, k64, v64, do64)
    return {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}


def group_slices(hq, hkv, b, kv):
    g = hq // hkv
    return slice(kv * g, kv * g + g)


def compare_group(gpu: dict, q, k, v, do, b, kv):
    """Oracle for one (batch, KV head) group vs the matching slices of GPU outputs.
    Returns {name: rel_fro}."""
    q64, k64, v64, do64 = (to64(x[b : b + 1]) for x in (q, k, v, do))
    ref = oracle.group_reference(q64, k64, v64, do64, 0, kv)
    hs = group_slices(q.shape[2], k.shape[2], b, kv)
    got = {
        "O": to64(gpu["O"][b, :, hs]),
        "LSE": to64(gpu["LSE"][b, hs]),
        "dQ": to64(gpu["dQ"][b, :, hs]),
        "dK": to64(gpu["dK"][b, :, kv]),
        "dV": to64(gpu["dV"][b, :, kv]),
    }
    return {n: rel_fro(got[n], ref[n]) for n in got}
