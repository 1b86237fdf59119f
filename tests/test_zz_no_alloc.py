"""The allocation-free backward (rca_attn_bwd_noalloc) against rca_attn_bwd.

rca_attn_bwd_noalloc serves callers that cannot allocate device memory at call
time: its scratch is an array built into the library. This file is collected
last on purpose, so that a failure here comes after every other test has run;
it also passes on its own in a fresh process (the first call does the set-up).
"""

import ctypes
import time

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300 import _native
from causal_head_attention_gb300.inputs import make_inputs, small
from tests.parity import TOL, rel_fro, to64

pytestmark = pytest.mark.gpu

LIMIT = 40 << 20  # bytes of built-in scratch


def _check_against_workspace_path(dt, shape, seed, calls=2):
    B, Hq, Hkv, T, Dh = shape
    w = small("noalloc", B, Hq, Hkv, T, Dh, dt, seed=seed)
    q, k, v, do = (x.cuda() for x in make_inputs(w))
    out, lse = rca.attention_forward(q, k, v)
    dq_ref, dk_ref, dv_ref = rca.attention_backward(q, k, v, out, lse, do)
    rca.rca_stream_status()
    for _ in range(calls):  # the shared scratch keeps the previous call's contents
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rca.rca_attn_bwd_noalloc(q, k, v, out, lse, do, dq, dk, dv)
        torch.cuda.synchronize()
        rca.rca_stream_status()
        tol = TOL[dt]
        assert rel_fro(to64(dq), to64(dq_ref)) <= tol["dQ"]
        assert rel_fro(to64(dk), to64(dk_ref)) <= tol["dK"]
        assert rel_fro(to64(dv), to64(dv_ref)) <= tol["dV"]


@pytest.mark.parametrize("dt,shape", [("bf16", (2, 4, 2, 333, 64)), ("fp32", (1, 2, 1, 200, 32))])
def test_noalloc_matches_workspace_backward_twice(dt, shape):
    _check_against_workspace_path(dt, shape, seed=11)


def test_noalloc_layouts_in_sequence_near_the_limit():
    """A call whose scratch nearly fills the array (fp32 storage, with its bf16
    hi/lo copies), then a smaller call with another scratch layout (bf16, head
    width 128, GQA), then the large one again: stale contents of the other
    layout must not leak into any result."""
    big = (2, 12, 3, 1920, 64)
    need = _native.rca_attn_bwd_workspace_size(*big, _native.RCA_F32_TF32)
    assert LIMIT - (1 << 20) < need <= LIMIT
    _check_against_workspace_path("fp32", big, seed=21, calls=1)
    _check_against_workspace_path("bf16", (1, 8, 2, 700, 128), seed=22, calls=1)
    _check_against_workspace_path("fp32", big, seed=23, calls=1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _native.lib()
    fake = ctypes.c_void_p(4096)  # rejected before any pointer is used
    st = lib.rca_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  8, 32, 32, 8192, 128, 1, ctypes.c_void_p(0))
    assert st == _native.RCA_ERR_INVALID_ARGUMENT
    assert "built-in scratch" in lib.rca_last_error().decode()
    # the first size past the limit, one 128-row tile beyond the near-limit case
    T = 1920
    while lib.rca_attn_bwd_workspace_size(2, 12, 3, T, 64, 0) <= LIMIT:
        T += 128
    st = lib.rca_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                  2, 12, 3, T, 64, 0, ctypes.c_void_p(0))
    assert st == _native.RCA_ERR_INVALID_ARGUMENT


def test_noalloc_device_timeout_is_reported():
    """A bounded device wait that runs out, recorded in the allocation-free
    path's own status word, comes back through rca_stream_status; the word is
    cleared and the entry point still works afterwards."""
    old = rca.rca_set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        t0 = time.perf_counter()
        rca.rca_selftest_noalloc_timeout()
        with pytest.raises(rca.RcaError) as e:
            rca.rca_stream_status()
        assert e.value.status == _native.RCA_ERR_DEVICE_TIMEOUT
        assert time.perf_counter() - t0 < 30.0
        rca.rca_stream_status()  # cleared
    finally:
        rca.rca_set_wait_timeout_ns(old)
    _check_against_workspace_path("bf16", (1, 2, 2, 130, 64), seed=12, calls=1)
