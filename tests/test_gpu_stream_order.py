"""Stream order of the training-step kernels, which the library launches with
programmatic dependent launch (each may be scheduled while the kernel before
it in the stream is still finishing, and waits for it before touching memory).

Steps run back to back on one stream with nothing between the launches but
ordinary torch kernels that overwrite the inputs and copy the outputs away;
every step's results must equal those of the same step run on its own with
the device synchronised around it. The workloads have more work items than
SMs, so the persistent CTAs are still running items when the next kernel is
launched.
"""

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300.inputs import make_inputs, small
from tests.parity import rel_fro, to64

pytestmark = pytest.mark.gpu

CASES = [
    ("order_bf16_dh64", 2, 16, 16, 1024, 64, "bf16"),
    ("order_bf16_dh128_gqa", 2, 8, 4, 2560, 128, "bf16"),
    ("order_fp32_dh64", 2, 12, 12, 1024, 64, "fp32"),
]


def step(bufs, outs, ws, Hkv, stream):
    q, k, v, do = bufs
    out, lse, dq, dk, dv = outs
    rca.rca_attn_fwd(q, k, v, out, lse, stream)
    rca.rca_attn_bwd_preprocess(out, lse, do, ws, Hkv=Hkv, stream=stream)
    rca.rca_attn_bwd_main(q, k, v, do, dk, dv, ws, stream)
    rca.rca_attn_bwd_dq_convert(dq, ws, Hkv=Hkv, stream=stream)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_back_to_back_steps_see_their_own_inputs(case):
    name, B, Hq, Hkv, T, Dh, dt = case
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    sets = [tuple(x.to(dev) for x in make_inputs(small(name, B, Hq, Hkv, T, Dh, dt, seed=s))) for s in (11, 12)]
    bufs = tuple(torch.empty_like(x) for x in sets[0])
    outs = (torch.empty_like(bufs[0]), torch.empty((B, Hq, T), dtype=torch.float32, device=dev),
            torch.empty_like(bufs[0]), torch.empty_like(bufs[1]), torch.empty_like(bufs[2]))
    ws = rca.workspace_for(bufs[0], bufs[1])

    # Each input set on its own, synchronised before and after.
    ref = []
    for s in sets:
        torch.cuda.synchronize(dev)
        for b, x in zip(bufs, s):
            b.copy_(x)
        torch.cuda.synchronize(dev)
        step(bufs, outs, ws, Hkv, stream)
        torch.cuda.synchronize(dev)
        rca.rca_stream_status(stream)
        ref.append(tuple(o.clone() for o in outs))

    # Six steps back to back, alternating the input sets, no synchronisation.
    got = []
    for i in range(6):
        for b, x in zip(bufs, sets[i % 2]):
            b.copy_(x)
        step(bufs, outs, ws, Hkv, stream)
        got.append(tuple(o.clone() for o in outs))
    torch.cuda.synchronize(dev)
    rca.rca_stream_status(stream)

    for i, g in enumerate(got):
        r = ref[i % 2]
        # The forward, dK and dV are deterministic: bit-identical.
        for n, a, b in zip(("O", "LSE", "dK", "dV"), (g[0], g[1], g[3], g[4]), (r[0], r[1], r[3], r[4])):
            assert torch.equal(a, b), f"step {i}: {n} differs from the synchronised run"
        # dQ partials are added by bulk reductions in arrival order: equal up
        # to the rounding of the fp32 sums.
        e = rel_fro(to64(g[2]), to64(r[2]))
        assert e < 1e-3, f"step {i}: dQ rel err {e:.2e} against the synchronised run"


def test_consumer_kernel_right_after_the_forward():
    """An ordinary kernel queued right after the forward reads its finished output."""
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    q, k, v, _ = (x.to(dev) for x in make_inputs(small("order_consumer", 2, 16, 16, 1024, 64, "bf16", seed=5)))
    out = torch.empty_like(q)
    lse = torch.empty((2, 16, 1024), dtype=torch.float32, device=dev)
    rca.rca_attn_fwd(q, k, v, out, lse, stream)
    torch.cuda.synchronize(dev)
    want_o, want_l = out.clone(), lse.clone()
    sums = []
    for _ in range(4):
        out.zero_()
        lse.zero_()
        rca.rca_attn_fwd(q, k, v, out, lse, stream)
        sums.append((out.float().sum(), lse.sum(), out.clone(), lse.clone()))
    torch.cuda.synchronize(dev)
    rca.rca_stream_status(stream)
    for s_o, s_l, o, l in sums:
        assert torch.equal(o, want_o) and torch.equal(l, want_l)
        assert s_o.item() == want_o.float().sum().item() and s_l.item() == want_l.sum().item()
