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

# Absolute floor (RMS per element) added to the denominator of the relative
# error. It only matters where the reference vanishes identically, e.g. dQ and
# dK at T = 1, which are exactly 0 in exact arithmetic (the oracle returns
# ~1e-17 from rounding, so a pure ratio would be meaningless there).
ATOL_RMS = 1e-5


def rel_fro(got, ref, atol_rms: float = ATOL_RMS) -> float:
    """||got - ref||_F / (||ref||_F + atol_rms * sqrt(n)), in fp64."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref) + atol_rms * np.sqrt(max(ref.size, 1))
    return float(np.linalg.norm(got - ref) / den)


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
