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


# Per-row bounds. A row is one query row of O / dQ, one key row of dK / dV
# (Dh elements). Whole-tensor norms can hide a few wrong rows; every row is
# therefore also held to ROW_FACTOR times the whole-tensor bound, relative to
# max(||ref_row||, ROW_FLOOR * rms row norm of the tensor). The floor keeps
# rows whose exact value is (near) zero, e.g. dQ of query 0, from turning
# rounding noise into a large relative error. A stale, shifted, zeroed or
# partly written row errs by O(1) and a single wrong element by about
# 1/sqrt(Dh) of the row, so both stay far above these bounds, while rounding
# (bf16 P and dS: 2^-9 per element) puts ordinary rows near the whole-tensor
# error. LSE is checked elementwise. With bf16 storage the scores are exact
# products accumulated in fp32, so LSE carries only ~1e-6 (fp32 sums,
# hardware exp2/log2). With fp32 storage the scores are TF32 products: each
# operand keeps 10 of its 23 mantissa bits (relative error up to 2^-10), so a
# score is off by up to 2^-9 * scale * sum_d |q_d k_d|, about 1e-3 to 1e-2 at
# unit-variance inputs, and LSE follows its largest scores. A wrong row is off
# by far more than either bound.
ROW_FACTOR = 5.0
ROW_FLOOR = 0.1
LSE_ABS = {"bf16": 1e-3, "fp32": 1e-2}
# fp32 storage: a row of O inherits the TF32 error of that row's largest
# scores (the same 2^-9 * scale * sum_d |q_d k_d| as LSE), which does not
# average out over the row's keys; its per-row bound is that size, 1e-2.
ROW_TOL = {dt: {n: ROW_FACTOR * t for n, t in tol.items()} for dt, tol in TOL.items()}
ROW_TOL["fp32"]["O"] = 1e-2


def row_violations(got, ref, tol, floor=ROW_FLOOR):
    """Rows (flattened index over all but the last axis) whose relative error
    exceeds tol; returns (indices, worst relative error)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got.shape[-1]
    g2, r2 = got.reshape(-1, d), ref.reshape(-1, d)
    err = np.linalg.norm(g2 - r2, axis=1)
    rn = np.linalg.norm(r2, axis=1)
    rms = float(np.sqrt(np.mean(rn * rn))) if rn.size else 0.0
    den = np.maximum(rn, floor * rms)
    den = np.where(den > 0, den, 1.0)
    rel = err / den
    return np.flatnonzero(rel > tol), float(rel.max()) if rel.size else 0.0


def check_rows(label, got: dict, ref: dict, dt: str, grad_ref: dict | None = None, skip=()):
    """Per-row checks of O, dQ, dK, dV and the elementwise LSE check; raises
    AssertionError naming the first offending rows.

    grad_ref: reference gradients of the backward evaluated on the arguments it
    was actually handed, i.e. with D = rowsum(dO * out) formed from the stored
    forward output (its bf16 rounding makes sum_j dS[i,j] differ from 0 by
    about 2^-9 |D_i|, which adds -scale * delta_i * (P K)_i to dQ row i: a
    real part of the method's answer, large against short or near one-hot
    rows). The whole-tensor bounds stay against the exact oracle.
    skip: outputs not checked per row (dQ, dK at T = 1, which vanish exactly)."""
    msgs = []
    for n in ("O", "dQ", "dK", "dV"):
        if n not in got or n in skip:
            continue
        r = grad_ref[n] if (grad_ref is not None and n in grad_ref) else ref[n]
        rt = ROW_TOL[dt][n]
        idx, worst = row_violations(got[n], r, rt)
        if idx.size:
            shape = np.asarray(ref[n]).shape[:-1]
            first = [tuple(int(c) for c in np.unravel_index(i, shape)) for i in idx[:4]]
            msgs.append(f"{n}: {idx.size} rows above {rt:.3g} (worst {worst:.3g}), e.g. {first}")
    if "LSE" in got:
        g, r = np.asarray(got["LSE"], dtype=np.float64), np.asarray(ref["LSE"], dtype=np.float64)
        e = np.abs(g - r)
        if not np.all(e <= LSE_ABS[dt]):
            bad = np.argwhere(e > LSE_ABS[dt])[:4].tolist()
            msgs.append(f"LSE: max abs err {e.max():.3g} at e.g. {bad}")
    assert not msgs, f"{label}: " + "; ".join(msgs)


def worst_rows(got: dict, ref: dict, grad_ref: dict | None = None) -> dict:
    """Worst per-row relative error of each output (for reporting margins)."""
    out = {}
    for n in ("O", "dQ", "dK", "dV"):
        if n in got:
            r = grad_ref[n] if (grad_ref is not None and n in grad_ref) else ref[n]
            out[n] = row_violations(got[n], r, np.inf)[1]
    if "LSE" in got:
        out["LSE_abs"] = float(np.max(np.abs(np.asarray(got["LSE"], np.float64) - np.asarray(ref["LSE"], np.float64))))
    return out


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


def grad_reference(q, k, v, do, out):
    """The oracle backward handed the stored forward output `out` (D reads it):
    dict of fp64 dQ, dK, dV."""
    q64, k64, v64, do64, o64 = (to64(x) for x in (q, k, v, do, out))
    dq, dk, dv = oracle.attention_backward(q64, k64, v64, do64, o=o64)
    return {"dQ": dq, "dK": dk, "dV": dv}


def group_slices(hq, hkv, b, kv):
    g = hq // hkv
    return slice(kv * g, kv * g + g)


def group_outputs(gpu: dict, q, k, v, do, b, kv):
    """Oracle for one (batch, KV head) group and the matching slices of the GPU
    outputs: (got, ref, grad_ref), dicts of fp64 arrays with the same shapes;
    grad_ref is the backward handed the GPU's stored output."""
    q64, k64, v64, do64 = (to64(x[b : b + 1]) for x in (q, k, v, do))
    o64 = to64(gpu["O"][b : b + 1])
    ref = oracle.group_reference(q64, k64, v64, do64, 0, kv, o=o64)
    hs = group_slices(q.shape[2], k.shape[2], b, kv)
    got = {
        "O": to64(gpu["O"][b, :, hs]),
        "LSE": to64(gpu["LSE"][b, hs]),
        "dQ": to64(gpu["dQ"][b, :, hs]),
        "dK": to64(gpu["dK"][b, :, kv]),
        "dV": to64(gpu["dV"][b, :, kv]),
    }
    grad_ref = {n: np.asarray(ref["given_o"][n], dtype=np.float64).reshape(got[n].shape)
                for n in ("dQ", "dK", "dV")}
    return got, {n: np.asarray(ref[n], dtype=np.float64).reshape(got[n].shape) for n in got}, grad_ref


def compare_group(gpu: dict, q, k, v, do, b, kv):
    """Oracle for one (batch, KV head) group vs the matching slices of GPU outputs.
    Returns {name: rel_fro}."""
    got, ref, _ = group_outputs(gpu, q, k, v, do, b, kv)
    return {n: rel_fro(got[n], ref[n]) for n in got}
