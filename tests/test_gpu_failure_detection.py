"""Failure detection on the GPU without a fault: a kernel waits on a barrier
that nothing completes; the time-bounded wait gives up, the status word reports
RCA_ERR_DEVICE_TIMEOUT through rca_stream_status, and the context stays usable."""

import time

import pytest
import torch

import causal_head_attention_gb300 as rca
from causal_head_attention_gb300 import _native
from causal_head_attention_gb300.inputs import make_inputs, small

pytestmark = pytest.mark.gpu


def test_device_wait_times_out_and_context_survives():
    old = rca.rca_set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        t0 = time.perf_counter()
        rca.rca_selftest_device_timeout()
        with pytest.raises(rca.RcaError) as e:
            rca.rca_stream_status()
        assert e.value.status == _native.RCA_ERR_DEVICE_TIMEOUT
        assert time.perf_counter() - t0 < 30.0
        # the status word was cleared and the context still works
        rca.rca_stream_status()
        w = small("after_timeout", 1, 2, 2, 130, 64, "bf16", seed=9)
        q, k, v, _ = (x.cuda() for x in make_inputs(w))
        out, lse = rca.attention_forward(q, k, v)
        rca.rca_stream_status()
        assert torch.isfinite(out.float()).all()
    finally:
        rca.rca_set_wait_timeout_ns(old)
