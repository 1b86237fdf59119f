"""The training step (forward + backward through the C ABI) captured in a CUDA
graph and replayed: the library's kernels are launched with programmatic
dependent launch, which a graph records as programmatic edges. Each replay
reads the current contents of the captured input buffers; its outputs must
equal those of an eager run on the same inputs (bit for bit, but for dQ, whose
fp32 partials are added in arrival order)."""

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300.inputs import make_inputs, small
from tests.parity import rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize(
    "case",
    [("graph_bf16_dh64", 2, 16, 16, 1024, 64, "bf16"), ("graph_bf16_dh128_gqa", 1, 8, 2, 1000, 128, "bf16")],
    ids=lambda c: c[0],
)
def test_captured_step_replays_on_new_inputs(case):
    name, B, Hq, Hkv, T, Dh, dt = case
    dev = torch.device("cuda:0")
    sets = [tuple(x.to(dev) for x in make_inputs(small(name, B, Hq, Hkv, T, Dh, dt, seed=s))) for s in (31, 32, 33)]
    q, k, v, do = (torch.empty_like(x) for x in sets[0])
    out, lse = torch.empty_like(q), torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = rca.workspace_for(q, k)

    def step(stream):
        rca.rca_attn_fwd(q, k, v, out, lse, stream)
        rca.rca_attn_bwd(q, k, v, out, lse, do, dq, dk, dv, ws, stream)

    def eager(inputs):
        for b, x in zip((q, k, v, do), inputs):
            b.copy_(x)
        step(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        rca.rca_stream_status()
        return tuple(t.clone() for t in (out, lse, dq, dk, dv))

    want = [eager(s) for s in sets]  # also the warm-up: first-call set-up happens outside the capture

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    torch.cuda.current_stream(dev).wait_stream(side)

    for i in (1, 2, 0, 1):
        for b, x in zip((q, k, v, do), sets[i]):
            b.copy_(x)
        for t in (out, lse, dq, dk, dv):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize(dev)
        rca.rca_stream_status()
        w = want[i]
        for n, a, b in zip(("O", "LSE", "dK", "dV"), (out, lse, dk, dv), (w[0], w[1], w[3], w[4])):
            assert torch.equal(a, b), f"replay on input set {i}: {n} differs from the eager run"
        e = rel_fro(to64(dq), to64(w[2]))
        assert e < 1e-3, f"replay on input set {i}: dQ rel err {e:.2e} against the eager run"
