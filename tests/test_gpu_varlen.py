"""GPU parity of padded / variable-length batches (right padding, per-sequence
lengths on the device) against the fp64 oracle.

Real rows are compared with the parity tolerances of the full-sequence tests;
padding rows must be exactly zero (LSE -inf), as must every gradient row at a
padding position; changing the (finite) contents of padding positions must
not change any real output.
"""

import zlib

import numpy as np
import pytest
import torch

import causal_head_attention_gb300 as rca
import oracle
from causal_head_attention_gb300.inputs import HEADLINE, make_inputs, small
from tests.parity import TOL, rel_fro, to64

pytestmark = pytest.mark.gpu


def run(q, k, v, do, lens):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    ld = torch.tensor(lens, dtype=torch.int32, device=dev)
    out, lse = rca.attention_forward_varlen(qd, kd, vd, ld)
    dq, dk, dv = rca.attention_backward_varlen(qd, kd, vd, out, lse, dod, ld)
    rca.rca_stream_status()
    return out, lse, dq, dk, dv


def real_mask(lens, T):
    return np.arange(T)[None, :] < np.asarray(lens)[:, None]  # [B, T]


CASES = [
    # name, B, Hq, Hkv, T, Dh, dtype, lens
    ("vl_bf16_dh64_gqa", 4, 4, 2, 300, 64, "bf16", [300, 129, 1, 0]),
    ("vl_bf16_dh128", 3, 2, 2, 257, 128, "bf16", [128, 256, 200]),
    # head width 128 with a group of 4: the 64-row sub-tile backward over a planned work list
    # (a length ending inside the first and inside the second half of a 128-row tile)
    ("vl_bf16_dh128_gqa", 3, 8, 2, 600, 128, "bf16", [600, 129, 65]),
    ("vl_bf16_dh32", 2, 4, 1, 130, 32, "bf16", [127, 65]),
    ("vl_fp32_dh64", 3, 2, 2, 200, 64, "fp32", [200, 77, 128]),
    ("vl_fp32_dh16_gqa", 2, 4, 2, 140, 16, "fp32", [3, 140]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_varlen_matches_oracle(case):
    name, B, Hq, Hkv, T, Dh, dt, lens = case
    w = small(name, B, Hq, Hkv, T, Dh, dt, seed=zlib.crc32(name.encode()) % 1000)
    q, k, v, do = make_inputs(w)
    out, lse, dq, dk, dv = run(q, k, v, do, lens)
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    o_ref, l_ref = oracle.attention_forward_varlen(q64, k64, v64, lens)
    g_ref = oracle.attention_backward_varlen(q64, k64, v64, do64, lens)
    m = real_mask(lens, T)
    got = {"O": to64(out), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
    ref = {"O": o_ref, "dQ": g_ref[0], "dK": g_ref[1], "dV": g_ref[2]}
    for n in got:
        assert np.all(got[n][~m] == 0), f"{name}: {n} nonzero at padding"
        assert rel_fro(got[n][m], ref[n][m]) <= TOL[dt][n], f"{name}: {n} {rel_fro(got[n][m], ref[n][m]):.3g}"
    lg = to64(lse)
    lm = np.broadcast_to(m[:, None, :], lg.shape)
    assert np.all(np.isneginf(lg[~lm])), f"{name}: LSE at padding is not -inf"
    assert rel_fro(lg[lm], l_ref[lm]) <= TOL[dt]["LSE"]


def test_padding_contents_do_not_reach_real_outputs():
    w = small("vl_invariance", 3, 4, 2, 260, 64, "bf16", seed=41)
    q, k, v, do = make_inputs(w)
    lens = [260, 100, 5]
    a = run(q, k, v, do, lens)
    g = torch.Generator().manual_seed(42)
    q2, k2, v2, do2 = (x.clone() for x in (q, k, v, do))
    for b, n in enumerate(lens):
        for x in (q2, k2, v2, do2):
            x[b, n:] = (torch.randn(x[b, n:].shape, generator=g) * 50).to(x.dtype)
    b_ = run(q2, k2, v2, do2, lens)
    for name, x, y in zip(("O", "LSE", "dQ", "dK", "dV"), a, b_):
        if name == "dQ":  # fp32 atomics: summation order may differ between runs
            assert rel_fro(to64(x), to64(y)) < 1e-6
        else:
            assert torch.equal(x, y), name


def test_full_length_equals_dense_path():
    w = small("vl_dense", 2, 4, 4, 192, 64, "bf16", seed=43)
    q, k, v, do = make_inputs(w)
    out, lse, dq, dk, dv = run(q, k, v, do, [192, 192])
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out_d, lse_d = rca.attention_forward(qd, kd, vd)
    assert torch.equal(out, out_d) and torch.equal(lse, lse_d)


def test_headline_random_lengths_sampled():
    q, k, v, do = make_inputs(HEADLINE)
    lens = [2048, 1000, 1, 1537]
    out, lse, dq, dk, dv = run(q, k, v, do, lens)
    for b in range(HEADLINE.B):
        n = lens[b]
        assert torch.all(out[b, n:] == 0) and torch.all(dq[b, n:] == 0) and torch.all(dk[b, n:] == 0)
    for b, kv in ((1, 0), (3, HEADLINE.Hkv - 1)):
        n = lens[b]
        ref = oracle.group_reference(to64(q[:, :n]), to64(k[:, :n]), to64(v[:, :n]), to64(do[:, :n]), b, kv)
        g = HEADLINE.Hq // HEADLINE.Hkv
        assert rel_fro(to64(out[b, :n, kv * g:(kv + 1) * g]), ref["O"]) <= TOL["bf16"]["O"]
        assert rel_fro(to64(dk[b, :n, kv]), ref["dK"]) <= TOL["bf16"]["dK"]
        assert rel_fro(to64(dv[b, :n, kv]), ref["dV"]) <= TOL["bf16"]["dV"]
        assert rel_fro(to64(dq[b, :n, kv * g:(kv + 1) * g]), ref["dQ"]) <= TOL["bf16"]["dQ"]


def test_bad_length_is_reported():
    w = small("vl_bad", 2, 2, 2, 64, 64, "bf16", seed=44)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out, lse = rca.attention_forward_varlen(qd, kd, vd, torch.tensor([64, 65], dtype=torch.int32, device=dev))
    with pytest.raises(rca.RcaError) as ei:
        rca.rca_stream_status()
    assert ei.value.status == 5
    out2, _ = rca.attention_forward_varlen(qd, kd, vd, torch.tensor([64, 64], dtype=torch.int32, device=dev))
    rca.rca_stream_status()
    assert torch.equal(out, out2)  # clamped to T


def test_maximum_batch_sampled():
    """4096 sequences (the most one call takes) of one tile each: the planner
    sorts and lists them all on the device. Padding is exactly zero everywhere;
    sampled sequences, including empty and full ones, match the oracle."""
    B, T = 4096, 128
    w = small("vl_maxbatch", B, 2, 1, T, 64, "bf16", seed=45)
    q, k, v, do = make_inputs(w)
    g = torch.Generator().manual_seed(46)
    lens = torch.randint(0, T + 1, (B,), generator=g)
    lens[0], lens[1], lens[B - 1] = 0, T, 1
    lens = lens.tolist()
    out, lse, dq, dk, dv = run(q, k, v, do, lens)
    m = real_mask(lens, T)
    for name, x in (("O", out), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert torch.all(x.float().cpu()[torch.from_numpy(~m)] == 0), f"{name} nonzero at padding"
    sel = [0, 1, 2, 2047, B - 2, B - 1]
    q64, k64, v64, do64 = (to64(x)[sel] for x in (q, k, v, do))
    ls = [lens[i] for i in sel]
    o_ref, l_ref = oracle.attention_forward_varlen(q64, k64, v64, ls)
    g_ref = oracle.attention_backward_varlen(q64, k64, v64, do64, ls)
    ms = real_mask(ls, T)
    got = {"O": to64(out)[sel], "dQ": to64(dq)[sel], "dK": to64(dk)[sel], "dV": to64(dv)[sel]}
    ref = {"O": o_ref, "dQ": g_ref[0], "dK": g_ref[1], "dV": g_ref[2]}
    for n in got:
        assert rel_fro(got[n][ms], ref[n][ms]) <= TOL["bf16"][n], n
    lg = to64(lse)[sel]
    lm = np.broadcast_to(ms[:, None, :], lg.shape)
    assert np.all(np.isneginf(lg[~lm])) and rel_fro(lg[lm], l_ref[lm]) <= TOL["bf16"]["LSE"]
