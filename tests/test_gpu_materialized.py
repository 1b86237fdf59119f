"""GPU parity of the materialized path (probabilities returned and kept for the
VJP) through the C ABI, against the fp64 oracle, and a full-size cross-check
of the memory-linear kernels against it.

Tolerances (derived from the arithmetic): the scores are exact bf16 products
accumulated in fp32 (or fp32 products), the softmax and the products over T
run in fp32, so against the oracle on the same stored inputs the
probabilities and LSE carry a few fp32 roundings: |dP| <= 2e-6 + 2e-5 P,
|dLSE| <= 2e-5 + 1e-6 |LSE|. Outputs in bf16 add one rounding (2^-9
relative): |dO| <= 2^-8 |O| + 1e-5 elementwise and 3e-3 relative Frobenius for
the gradients; fp32 storage: 2e-5 relative Frobenius for all outputs.
"""

import zlib

import numpy as np
import pytest
import torch

import causal_head_attention_gb300 as rca
import oracle
from causal_head_attention_gb300.inputs import HEADLINE, make_inputs, small
from tests.parity import rel_fro, to64

pytestmark = pytest.mark.gpu

GRAD_TOL = {"bf16": 3e-3, "fp32": 2e-5}


def gpu_mat(q, k, v, do, dp=None):
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in (q, k, v, do))
    out, probs, lse = rca.materialized_forward(q, k, v)
    dq, dk, dv = rca.materialized_backward(q, k, v, probs, do, None if dp is None else dp.to(dev))
    rca.rca_stream_status()
    return out, probs, lse, dq, dk, dv


def check_probs(name, probs, lse, p_ref, l_ref):
    p, l = to64(probs), to64(lse)
    err = np.abs(p - p_ref)
    bad = err > 2e-6 + 2e-5 * np.abs(p_ref)
    assert not bad.any(), f"{name}: probs off at {np.argwhere(bad)[:4].tolist()}, max {err.max():.3g}"
    t = p.shape[-1]
    assert np.all(p[..., np.triu_indices(t, 1)[0], np.triu_indices(t, 1)[1]] == 0), f"{name}: nonzero above diagonal"
    lerr = np.abs(l - l_ref)
    assert np.all(lerr <= 2e-5 + 1e-6 * np.abs(l_ref)), f"{name}: LSE max err {lerr.max():.3g}"


CASES = [
    # name, B, Hq, Hkv, T, Dh, dtype
    ("bf16_dh64_gqa", 2, 4, 2, 96, 64, "bf16"),
    ("bf16_dh128_t_odd", 1, 2, 2, 77, 128, "bf16"),
    ("bf16_dh16", 1, 3, 1, 130, 16, "bf16"),
    ("fp32_dh32_gqa", 1, 4, 1, 64, 32, "fp32"),
    ("fp32_dh128", 1, 2, 2, 50, 128, "fp32"),
    ("bf16_t1", 2, 2, 2, 1, 64, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("with_dp", [False, True], ids=["dO", "dO+dP"])
def test_small_every_output(case, with_dp):
    name, B, Hq, Hkv, T, Dh, dt = case
    w = small(name, B, Hq, Hkv, T, Dh, dt, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v, do = make_inputs(w)
    dp = torch.randn((B, Hq, T, T), generator=torch.Generator().manual_seed(7)) if with_dp else None
    out, probs, lse, dq, dk, dv = gpu_mat(q, k, v, do, dp)
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    o_ref, p_ref, l_ref = oracle.attention_probs(q64, k64, v64)
    check_probs(name, probs, lse, p_ref, l_ref)
    o = to64(out)
    if dt == "bf16":
        err = np.abs(o - o_ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(o_ref) + 1e-5), f"{name}: O max err {err.max():.3g}"
    else:
        assert rel_fro(o, o_ref) <= GRAD_TOL["fp32"], name
    ref = oracle.materialized_backward(q64, k64, v64, do64, None if dp is None else dp.double().numpy())
    for nm, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        e = rel_fro(to64(got), r)
        if T == 1 and nm in ("dQ", "dK") and not with_dp:
            assert np.abs(to64(got)).max() < 1e-5, (name, nm)  # exactly zero in exact arithmetic
            continue
        assert e <= GRAD_TOL[dt], f"{name} {nm}: {e:.3g}"


# Mid-size shapes where every persistent CTA of the product kernels takes
# several items (score tiles, 128-row output blocks, 128-key output blocks).
MULTI = [
    # name, B, Hq, Hkv, T, Dh, dtype      score tiles / row items / column items
    ("bf16_dh32_gqa_multi", 4, 8, 4, 1300, 32, "bf16"),   # 2112 / 352 / 176
    ("fp32_dh64_multi", 2, 12, 12, 1000, 64, "fp32"),     # 864 / 192 / 192
]


@pytest.mark.parametrize("case", MULTI, ids=[c[0] for c in MULTI])
def test_multi_item_every_output(case):
    name, B, Hq, Hkv, T, Dh, dt = case
    w = small(name, B, Hq, Hkv, T, Dh, dt, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v, do = make_inputs(w)
    out, probs, lse, dq, dk, dv = gpu_mat(q, k, v, do)
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    o_ref, p_ref, l_ref = oracle.attention_probs(q64, k64, v64)
    check_probs(name, probs, lse, p_ref, l_ref)
    o = to64(out)
    if dt == "bf16":
        err = np.abs(o - o_ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(o_ref) + 1e-5), f"{name}: O max err {err.max():.3g}"
    else:
        assert rel_fro(o, o_ref) <= GRAD_TOL["fp32"], name
    ref = oracle.materialized_backward(q64, k64, v64, do64, None)
    for nm, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        e = rel_fro(to64(got), r)
        assert e <= GRAD_TOL[dt], f"{name} {nm}: {e:.3g}"


@pytest.mark.parametrize("case", [("nan_bf16_t300", 1, 2, 1, 300, 64, "bf16"), ("nan_fp32_t130", 1, 2, 2, 130, 32, "fp32")],
                         ids=lambda c: c[0])
def test_forward_writes_every_output_element(case):
    """Every element of out, probs and lse is written by the forward (the
    kept tiles by the probabilities pass, the rest of each row by the row
    pass): buffers filled with NaN beforehand must come back equal to the
    oracle, with exact zeros above the diagonal. T = 300 takes the 16-byte
    path, T = 130 the scalar one."""
    name, B, Hq, Hkv, T, Dh, dt = case
    q, k, v, _ = make_inputs(small(name, B, Hq, Hkv, T, Dh, dt, seed=5))
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out = torch.full_like(qd, float("nan"))
    probs = torch.full((B, Hq, T, T), float("nan"), device=dev)
    lse = torch.full((B, Hq, T), float("nan"), device=dev)
    ws = torch.full((rca.rca_attn_materialized_workspace_size(B, Hq, Hkv, T, Dh, qd.dtype),), 255, dtype=torch.uint8,
                    device=dev)
    rca.rca_attn_materialized_fwd(qd, kd, vd, out, probs, lse, ws)
    rca.rca_stream_status()
    q64, k64, v64 = (to64(x) for x in (q, k, v))
    o_ref, p_ref, l_ref = oracle.attention_probs(q64, k64, v64)
    check_probs(name, probs, lse, p_ref, l_ref)
    o = to64(out)
    assert not np.isnan(o).any(), f"{name}: unwritten output rows"
    if dt == "bf16":
        assert np.all(np.abs(o - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + 1e-5), name
    else:
        assert rel_fro(o, o_ref) <= GRAD_TOL["fp32"], name


def test_zero_dprobs_equals_none():
    w = small("mat_zero_dp", 1, 2, 2, 64, 64, "bf16", seed=3)
    q, k, v, do = make_inputs(w)
    a = gpu_mat(q, k, v, do, None)
    b = gpu_mat(q, k, v, do, torch.zeros((1, 2, 64, 64)))
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_headline_cross_check_with_flash():
    """The two GPU paths agree at full size; sampled heads match the oracle."""
    q, k, v, do = make_inputs(HEADLINE)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out_m, probs, lse_m = rca.materialized_forward(qd, kd, vd)
    dq_m, dk_m, dv_m = rca.materialized_backward(qd, kd, vd, probs, dod)
    out_f, lse_f = rca.attention_forward(qd, kd, vd)
    dq_f, dk_f, dv_f = rca.attention_backward(qd, kd, vd, out_f, lse_f, dod)
    rca.rca_stream_status()
    assert torch.allclose(lse_m, lse_f, atol=2e-3, rtol=0)
    for a, b in ((out_m, out_f), (dq_m, dq_f), (dk_m, dk_f), (dv_m, dv_f)):
        assert rel_fro(to64(a), to64(b)) < 1e-2
    # Sampled heads against the oracle, every element of their probabilities.
    for b_, h in ((0, 0), (HEADLINE.B - 1, HEADLINE.Hq - 1)):
        qh, kh, vh = (to64(x[b_, :, h]) for x in (q, k, v))
        o_ref, l_ref, p_ref = oracle.head_forward(qh, kh, vh, oracle.default_scale(HEADLINE.Dh))
        check_probs(f"headline b{b_} h{h}", probs[b_, h], lse_m[b_, h], p_ref, l_ref)
        err = np.abs(to64(out_m[b_, :, h]) - o_ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(o_ref) + 1e-5)


@pytest.mark.parametrize("T,tile", [(37, 1), (37, 5), (256, 128), (300, 128), (300, 1000), (130, 64)])
def test_causal_softmax_bwd_tiled(T, tile):
    """The tiled VJP: row i written for j < min(T, tile (i // tile + 1)), equal
    there to the whole-row VJP bit for bit and to the oracle within its bound;
    every other entry of grad left exactly as it was."""
    g = torch.Generator().manual_seed(1000 + T + tile)
    s = torch.randn((2, T, T), generator=g) * 3
    grad = torch.randn((2, T, T), generator=g)
    extra = torch.randn((2, T, T), generator=g)
    dev = torch.device("cuda:0")
    pd = s.to(dev)
    lse = torch.empty((2, T), device=dev)
    rca.rca_causal_softmax(pd, lse, 0.3)
    full, tiled, ed = grad.to(dev), grad.to(dev), extra.to(dev)
    rca.rca_causal_softmax_bwd(pd, full, ed, 0.3)
    rca.rca_causal_softmax_bwd_tiled(pd, tiled, ed, tile, 0.3)
    rca.rca_stream_status()
    i = torch.arange(T).view(T, 1)
    j = torch.arange(T).view(1, T)
    written = (j < torch.clamp((i // tile + 1) * tile, max=T)).expand(2, T, T)
    tc, fc = tiled.cpu(), full.cpu()
    assert torch.equal(tc[written], fc[written])
    assert torch.equal(tc[~written], grad[~written])
    d_ref = oracle.causal_softmax_vjp(to64(pd), (grad + extra).double().numpy(), 0.3)
    err = np.abs(to64(tc) - d_ref)[written.numpy()]
    assert np.all(err <= 1e-6 + 1e-4 * np.abs(d_ref[written.numpy()]))


@pytest.mark.parametrize("T", [1, 37, 256])
def test_causal_softmax_entries(T):
    """The fused causal softmax and its VJP on their own (in place)."""
    g = torch.Generator().manual_seed(T)
    s = torch.randn((3, T, T), generator=g) * 3
    grad = torch.randn((3, T, T), generator=g)
    extra = torch.randn((3, T, T), generator=g)
    dev = torch.device("cuda:0")
    sd, gd, ed = (x.to(dev) for x in (s, grad, extra))
    lse = torch.empty((3, T), device=dev)
    rca.rca_causal_softmax(sd, lse, 0.3)
    rca.rca_causal_softmax_bwd(sd, gd, ed, 0.3)
    rca.rca_stream_status()
    p_ref, l_ref = oracle.causal_softmax(s.double().numpy(), 0.3)
    check_probs(f"softmax T{T}", sd, lse, p_ref, l_ref)
    d_ref = oracle.causal_softmax_vjp(p_ref, (grad + extra).double().numpy(), 0.3)
    err = np.abs(to64(gd) - d_ref)
    assert np.all(err <= 1e-6 + 1e-4 * np.abs(d_ref)), f"softmax VJP T{T}: max err {err.max():.3g}"
