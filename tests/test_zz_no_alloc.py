"""The allocation-free backward (rca_attn_bwd_noalloc) against rca_attn_bwd.

rca_attn_bwd_noalloc serves callers that cannot allocate device memory at call
time: its scratch is an array built into the library. This file is collected
last on purpose, so that a failure here comes after every other test has run;
it also passes on its own in a fresh process (the first call does the set-up).
"""

import ctypes

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300 import _native
from causal_head_attention_gb300.inputs import make_inputs, small
from tests.parity import TOL, rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,shape", [("bf16", (2, 4, 2, 333, 64)), ("fp32", (1, 2, 1, 200, 32))])
def test_noalloc_matches_workspace_backward_twice(dt, shape):
    B, Hq, Hkv, T, Dh = shape
    w = small("noalloc", B, Hq, Hkv, T, Dh, dt, seed=11)
    q, k, v, do = (x.cuda() for x in make_inputs(w))
    out, lse = rca.attention_forward(q, k, v)
    dq_ref, dk_ref, dv_ref = rca.attention_backward(q, k, v, out, lse, do)
    rca.rca_stream_status()
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rca.rca_attn_bwd_noalloc(q, k, v, out, lse, do, dq, dk, dv)
        torch.cuda.synchronize()
        rca.rca_stream_status()
        tol = TOL[dt]
        assert rel_fro(to64(dq), to64(dq_ref)) <= tol["dQ"]
        assert rel_fro(to64(dk), to64(dk_ref)) <= tol["dK"]
        assert rel_fro(to64(dv), to64(dv_ref)) <= tol["dV"]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _native.lib()
    fake = ctypes.c_void_p(4096)  # rejected before any pointer is used
    st = lib.rca_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  8, 32, 32, 8192, 128, 1, ctypes.c_void_p(0))
    assert st == _native.RCA_ERR_INVALID_ARGUMENT
    assert "built-in scratch" in lib.rca_last_error().decode()
