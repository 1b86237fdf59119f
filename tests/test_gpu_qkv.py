"""GPU parity of the fused QKV layout: q, k, v read in place from one
[B, T, (Hq + 2*Hkv) * Dh] projection output and dq, dk, dv written in place into
one buffer of that shape. Same kernels as the separate-tensor path, so the
forward output is bit-identical to it; everything is also checked against the
fp64 oracle with the parity tolerances of the separate-tensor tests.
"""

import zlib

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300.inputs import HEADLINE, make_inputs, small
from tests.parity import TOL, full_reference, rel_fro, to64

pytestmark = pytest.mark.gpu


def fuse(q, k, v):
    B, T, Hq, Dh = q.shape
    Hkv = k.shape[2]
    return torch.cat([q.reshape(B, T, Hq * Dh), k.reshape(B, T, Hkv * Dh), v.reshape(B, T, Hkv * Dh)], dim=2)


def split(dqkv, Hq, Hkv, Dh):
    B, T, _ = dqkv.shape
    dq = dqkv[:, :, : Hq * Dh].reshape(B, T, Hq, Dh)
    dk = dqkv[:, :, Hq * Dh: (Hq + Hkv) * Dh].reshape(B, T, Hkv, Dh)
    dv = dqkv[:, :, (Hq + Hkv) * Dh:].reshape(B, T, Hkv, Dh)
    return dq, dk, dv


CASES = [
    ("qkv_bf16_dh64_gqa", 2, 4, 2, 300, 64, "bf16"),
    ("qkv_bf16_dh128", 1, 2, 2, 257, 128, "bf16"),
    ("qkv_bf16_dh32_gqa8", 1, 8, 1, 130, 32, "bf16"),
    ("qkv_fp32_dh64", 1, 2, 2, 200, 64, "fp32"),
    ("qkv_fp32_dh16_gqa", 2, 4, 1, 65, 16, "fp32"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_layout_matches_oracle_and_separate_path(case):
    name, B, Hq, Hkv, T, Dh, dt = case
    w = small(name, B, Hq, Hkv, T, Dh, dt, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    qkv = fuse(qd, kd, vd).contiguous()
    dout = dod.reshape(B, T, Hq * Dh)
    out, lse = rca.attention_forward_qkv(qkv, Hq, Hkv)
    dqkv = rca.attention_backward_qkv(qkv, Hq, Hkv, out, lse, dout)
    out_s, lse_s = rca.attention_forward(qd, kd, vd)
    rca.rca_stream_status()
    assert torch.equal(out.reshape(B, T, Hq, Dh), out_s) and torch.equal(lse, lse_s)
    ref = full_reference(q, k, v, do)
    dq, dk, dv = split(dqkv, Hq, Hkv, Dh)
    got = {"O": out.reshape(B, T, Hq, Dh), "LSE": lse, "dQ": dq, "dK": dk, "dV": dv}
    errs = {n: rel_fro(to64(got[n]), ref[n]) for n in ref}
    bad = {n: e for n, e in errs.items() if not e <= TOL[dt][n]}
    assert not bad, f"{name}: {errs}"


def test_autograd_node_on_fused_layout():
    w = small("qkv_autograd", 1, 4, 2, 160, 64, "bf16", seed=31)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qkv = fuse(*(x.to(dev) for x in (q, k, v))).contiguous().requires_grad_(True)
    out = rca.causal_attention_qkv(qkv, 4, 2)
    (out.float() * do.to(dev).reshape(1, 160, 256).float()).sum().backward()
    rca.rca_stream_status()
    ref = full_reference(q, k, v, do)
    dq, dk, dv = split(qkv.grad, 4, 2, 64)
    for n, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert rel_fro(to64(g), ref[n]) <= TOL["bf16"][n], n


def test_headline_fused_equals_separate():
    q, k, v, do = make_inputs(HEADLINE)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    B, T, H, Dh = q.shape
    qkv = fuse(qd, kd, vd).contiguous()
    out, lse = rca.attention_forward_qkv(qkv, H, H)
    dqkv = rca.attention_backward_qkv(qkv, H, H, out, lse, dod.reshape(B, T, H * Dh))
    out_s, lse_s = rca.attention_forward(qd, kd, vd)
    dq_s, dk_s, dv_s = rca.attention_backward(qd, kd, vd, out_s, lse_s, dod)
    rca.rca_stream_status()
    assert torch.equal(out.reshape(B, T, H, Dh), out_s)
    dq, dk, dv = split(dqkv, H, H, Dh)
    assert torch.equal(dk, dk_s) and torch.equal(dv, dv_s)
    assert rel_fro(to64(dq), to64(dq_s)) < 1e-3  # fp32 atomics: summation order differs
