"""GPU parity of paged decode attention (through the C ABI) against the fp64 oracle.

Small caches are compared element by element over every output: head widths
16..128, both storage dtypes, page sizes 1..256, query groups 1..16 (including
a group that is not a power of two; bf16 groups of 2 or more run on the tensor
cores, at every head width), lengths of one position, on page and
chunk boundaries (a chunk is 256 positions) and ragged. The two full-size decode
workloads run in the launch configuration the benchmark times and are compared
on sampled requests (the longest, the one-position one and a middle one), every
element of which the oracle computes exactly.

Tolerances (derived from the arithmetic): the kernel computes in fp32 from the
stored values, so against the oracle on the same stored values its error before
the final store is a few fp32 roundings (~1e-6 relative). A bf16 output then
adds one rounding to bf16 (at most 2^-9 relative): |got - ref| <= 2^-8 |ref| +
1e-4. fp32 storage: |got - ref| <= 2e-5 |ref| + 2e-5. LSE is fp32 in both:
|got - ref| <= 2e-5 + 1e-6 |ref| (one position more or less at L = 8192 moves
it by ~1e-4).
"""

import zlib

import numpy as np
import pytest
import torch

import causal_head_attention_gb300 as rca
import oracle
from causal_head_attention_gb300.inputs import DEC_GQA, DEC_MHA, PAGED_WORKLOADS, PagedWorkload, make_paged_inputs
from tests.parity import to64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2.0 ** -8, 1e-4), "fp32": (2e-5, 2e-5)}
LSE_TOL = (1e-6, 2e-5)


def run_gpu(q, kp, vp, table, lens):
    dev = torch.device("cuda:0")
    args = [x.to(dev) for x in (q, kp, vp, table, lens)]
    out, lse = rca.paged_decode(*args)
    rca.rca_stream_status()
    return out, lse


def check(name, dtype, out, lse, ref_o, ref_lse, rows=None):
    got_o, got_l = to64(out), to64(lse)
    if rows is not None:
        got_o, got_l = got_o[rows], got_l[rows]
    rt, at = TOL[dtype]
    err = np.abs(got_o - ref_o)
    bad = err > at + rt * np.abs(ref_o)
    assert not bad.any(), f"{name}: O off at {np.argwhere(bad)[:5].tolist()}, max err {err.max():.3g}"
    lerr = np.abs(got_l - ref_lse)
    lbad = lerr > LSE_TOL[1] + LSE_TOL[0] * np.abs(ref_lse)
    assert not lbad.any(), f"{name}: LSE off at {np.argwhere(lbad)[:5].tolist()}, max err {lerr.max():.3g}"


def oracle_of(q, kp, vp, table, lens, rows=None):
    q64, k64, v64 = to64(q), to64(kp), to64(vp)
    t, n = table.numpy(), lens.numpy()
    if rows is not None:
        q64, t, n = q64[rows], t[rows], n[rows]
    return oracle.paged_decode(q64, k64, v64, t, n)


SMALL = [
    # name, B, Hq, Hkv, Dh, page_size, max_len, dtype, lengths (None = drawn)
    ("small_gqa_bf16", 3, 4, 2, 64, 16, 300, "bf16", None),
    ("small_mha_fp32", 2, 4, 4, 32, 8, 100, "fp32", None),
    ("dh16_bf16_ps1", 3, 2, 2, 16, 1, 600, "bf16", [600, 1, 257]),
    ("dh16_fp32", 2, 3, 1, 16, 4, 520, "fp32", [520, 256]),
    ("dh32_bf16_g8", 2, 8, 1, 32, 32, 700, "bf16", [700, 512]),
    ("dh64_fp32_g2", 3, 4, 2, 64, 64, 1000, "fp32", [1000, 1, 513]),
    ("dh128_bf16_g4", 2, 8, 2, 128, 16, 1030, "bf16", [1030, 255]),
    ("dh128_fp32", 2, 2, 2, 128, 256, 800, "fp32", [800, 768]),
    ("g3_bf16", 2, 6, 2, 64, 16, 400, "bf16", [400, 17]),
    ("g16_bf16", 2, 16, 1, 64, 8, 300, "bf16", [300, 64]),
    ("one_chunk_only", 4, 4, 4, 64, 16, 256, "bf16", [256, 1, 16, 255]),
    ("all_len1", 5, 2, 1, 128, 4, 4, "bf16", [1, 1, 1, 1, 1]),
    # tensor-core kernel at Dh = 16 (8-byte K and 4-byte V fragment loads), pages
    # smaller than its 16-position block and pages holding whole blocks
    ("dh16_bf16_g4_ps2", 2, 8, 2, 16, 2, 300, "bf16", [300, 33]),
    ("dh16_bf16_g2_ps32", 3, 4, 2, 16, 32, 600, "bf16", [600, 1, 257]),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_every_output(case):
    name, B, Hq, Hkv, Dh, ps, max_len, dt, lengths = case
    w = PagedWorkload(name, B, Hq, Hkv, Dh, ps, max_len, dt, zlib.crc32(name.encode()) % 1000)
    q, kp, vp, table, lens = make_paged_inputs(w, lengths)
    out, lse = run_gpu(q, kp, vp, table, lens)
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens)
    check(name, dt, out, lse, ref_o, ref_l)


@pytest.mark.parametrize("w", [DEC_MHA, DEC_GQA], ids=[DEC_MHA.name, DEC_GQA.name])
def test_workload_sampled_requests(w):
    q, kp, vp, table, lens = make_paged_inputs(w)
    out, lse = run_gpu(q, kp, vp, table, lens)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    n = lens.numpy()
    rows = sorted({0, 1, w.B // 2, int(np.argmin(np.abs(n - 300)))})
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens, rows)
    check(w.name, w.dtype, out, lse, ref_o, ref_l, rows)


def test_page_placement_does_not_change_bits():
    """The same logical cache on other physical pages gives identical bits."""
    w = PagedWorkload("perm", 3, 8, 2, 128, 16, 900, "bf16", 21)
    q, kp, vp, table, lens = make_paged_inputs(w, [900, 300, 1])
    out0, lse0 = run_gpu(q, kp, vp, table, lens)
    g = torch.Generator().manual_seed(5)
    P = kp.shape[0]
    perm = torch.randperm(P + 11, generator=g)[:P]  # new slot of each old page, in a larger pool
    kq = torch.randn((P + 11,) + tuple(kp.shape[1:]), generator=g).to(kp.dtype)
    vq = torch.randn((P + 11,) + tuple(vp.shape[1:]), generator=g).to(vp.dtype)
    kq[perm] = kp
    vq[perm] = vp
    t2 = torch.where(table >= 0, perm[table.clamp(min=0).long()].to(torch.int32), table)
    out1, lse1 = run_gpu(q, kq, vq, t2, lens)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_repeatable():
    q, kp, vp, table, lens = make_paged_inputs(PAGED_WORKLOADS[0])
    a = run_gpu(q, kp, vp, table, lens)
    b = run_gpu(q, kp, vp, table, lens)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_graph_capture_replays():
    w = PagedWorkload("graph", 4, 8, 8, 64, 16, 1200, "bf16", 22)
    q, kp, vp, table, lens = (x.cuda() for x in make_paged_inputs(w))
    ws = torch.empty(rca.rca_paged_decode_workspace_size(4, 8, 8, 64, 16, table.shape[1], torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((4, 8), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rca.rca_paged_decode(q, kp, vp, table, lens, out, lse, ws, s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rca.rca_paged_decode(q, kp, vp, table, lens, out, lse, ws)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_of(q.cpu(), kp.cpu(), vp.cpu(), table.cpu(), lens.cpu())
    check("graph", "bf16", out, lse, ref_o, ref_l)


def test_bad_length_is_reported_and_isolated():
    """A length outside [1, max_pages * page_size] gives NaN for that request
    only and RCA_ERR_DEVICE_INVALID_INPUT; the other requests are exact."""
    w = PagedWorkload("badlen", 4, 4, 2, 64, 16, 600, "bf16", 23)
    q, kp, vp, table, lens = make_paged_inputs(w, [600, 40, 300, 2])
    bad = lens.clone()
    bad[1] = 0
    bad[3] = w.max_pages * w.page_size + 1
    dev = torch.device("cuda:0")
    out, lse = rca.paged_decode(*(x.to(dev) for x in (q, kp, vp, table, bad)))
    with pytest.raises(rca.RcaError) as ei:
        rca.rca_stream_status()
    assert ei.value.status == 5
    assert torch.isnan(out[1].float()).all() and torch.isnan(out[3].float()).all()
    assert torch.isnan(lse[1]).all() and torch.isnan(lse[3]).all()
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens, [0, 2])
    check("badlen", "bf16", out, lse, ref_o, ref_l, [0, 2])
    rca.rca_stream_status()  # the status was cleared by the report


def test_bad_page_id_is_reported_not_read():
    """A page ID outside [0, num_pages) is skipped (never dereferenced) and
    reported; requests that do not use it are exact."""
    w = PagedWorkload("badpage", 3, 4, 4, 64, 16, 400, "bf16", 24)
    q, kp, vp, table, lens = make_paged_inputs(w, [400, 100, 50])
    t2 = table.clone()
    t2[1, 2] = kp.shape[0] + 1000
    t2[1, 3] = -5
    dev = torch.device("cuda:0")
    out, lse = rca.paged_decode(*(x.to(dev) for x in (q, kp, vp, t2, lens)))
    with pytest.raises(rca.RcaError) as ei:
        rca.rca_stream_status()
    assert ei.value.status == 5
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens, [0, 2])
    check("badpage", "bf16", out, lse, ref_o, ref_l, [0, 2])
    rca.rca_stream_status()


def test_validation_errors_do_not_launch():
    q, kp, vp, table, lens = (x.cuda() for x in make_paged_inputs(PAGED_WORKLOADS[0]))
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    with pytest.raises(rca.RcaError) as ei:
        rca.rca_paged_decode(q, kp, vp, table, lens, out, lse, ws)
    assert ei.value.status == 1 and "workspace" in str(ei.value)
    rca.rca_stream_status()


@pytest.mark.parametrize("hq,hkv", [(4, 1), (2, 2)], ids=["tensor_core_g4", "cuda_core_g1"])
def test_maximum_batch(hq, hkv):
    """8192 requests (the most one call takes): every CTA rebuilds the request
    prefix sums over the whole batch in shared memory. Sampled requests are
    compared element by element; every output must be finite."""
    w = PagedWorkload(f"maxbatch_{hq}_{hkv}", 8192, hq, hkv, 16, 16, 300, "bf16", 25)
    q, kp, vp, table, lens = make_paged_inputs(w)
    out, lse = run_gpu(q, kp, vp, table, lens)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    n = lens.numpy()
    rows = sorted({0, 1, 4095, 4096, 8191, int(np.argmax(n)), int(np.argmin(n))})
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens, rows)
    check(w.name, "bf16", out, lse, ref_o, ref_l, rows)


def test_maximum_page_size():
    """Pages of 65536 positions (the largest page size) and a request spanning two."""
    w = PagedWorkload("maxpage", 2, 4, 2, 16, 65536, 70000, "bf16", 26)
    q, kp, vp, table, lens = make_paged_inputs(w, [70000, 5])
    out, lse = run_gpu(q, kp, vp, table, lens)
    ref_o, ref_l = oracle_of(q, kp, vp, table, lens)
    check("maxpage", "bf16", out, lse, ref_o, ref_l)
