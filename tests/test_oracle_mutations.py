"""Plant plausible mistakes in the oracle (on the CPU) and show the pins catch them.

Each mutant replaces one oracle function through monkeypatch; the pin that
should notice it is run and must fail.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as oa
from tests import test_oracle_pins as pins


def _backward_without_d(qh, kh, vh, oh, doh, p, scale):
    dv = p.T @ doh
    dp = doh @ vh.T
    ds = p * dp  # dropped the "- D" term
    return scale * ds @ kh, scale * ds.T @ qh, dv, np.zeros(len(qh))


def _backward_transposed_dk(qh, kh, vh, oh, doh, p, scale):
    dv = p.T @ doh
    dp = doh @ vh.T
    d = np.sum(doh * oh, axis=1)
    ds = p * (dp - d[:, None])
    return scale * ds @ kh, scale * ds @ qh, dv, d  # dS instead of dS^T


def _backward_wrong_sign(qh, kh, vh, oh, doh, p, scale):
    dv = p.T @ doh
    dp = doh @ vh.T
    d = np.sum(doh * oh, axis=1)
    ds = p * (dp + d[:, None])
    return scale * ds @ kh, scale * ds.T @ qh, dv, d


def _keep_strict(t):
    return np.tril(np.ones((t, t), dtype=bool), k=-1) | (np.arange(t)[:, None] == 0)


def _keep_anticausal(t):
    return np.triu(np.ones((t, t), dtype=bool))


@pytest.mark.parametrize("mutant", [_backward_without_d, _backward_transposed_dk, _backward_wrong_sign])
def test_fd_catches_backward_mutants(monkeypatch, mutant):
    monkeypatch.setattr(oa, "head_backward", mutant)
    with pytest.raises(AssertionError):
        pins.fd_check(1, 5, 2, 1, 4, seed=10)


@pytest.mark.parametrize("mask", [_keep_strict, _keep_anticausal])
def test_torch_check_catches_mask_mutants(monkeypatch, mask):
    monkeypatch.setattr(oa, "_causal_keep", mask)
    q, k, v, do = pins.rand_qkv(1, 9, 2, 2, 4, seed=1)
    o, _ = oracle.attention_forward(q, k, v)
    to, _, _, _ = pins.torch_sdpa(q, k, v, do)
    assert not np.allclose(o, to, rtol=1e-10, atol=1e-11)


def test_causality_catches_anticausal_mask(monkeypatch):
    monkeypatch.setattr(oa, "_causal_keep", _keep_anticausal)
    with pytest.raises(AssertionError):
        pins.test_causality_future_perturbation()


def test_closed_form_catches_missing_scale(monkeypatch):
    monkeypatch.setattr(oa, "default_scale", lambda dh: 1.0)
    with pytest.raises(AssertionError):
        pins.test_single_position_closed_form()


def test_torch_check_catches_wrong_head_map(monkeypatch):
    orig = oa.attention_forward

    def fwd_wrong_group(q, k, v, scale=None):
        b, t, hq, hkv, dh = oa._check_shapes(q, k, v)
        scale = oa.default_scale(dh) if scale is None else scale
        o = np.empty((b, t, hq, dh))
        lse = np.empty((b, hq, t))
        for bi in range(b):
            for h in range(hq):
                kv = h % hkv  # interleaved instead of consecutive groups
                oh, lh, _ = oa.head_forward(q[bi, :, h], k[bi, :, kv], v[bi, :, kv], scale)
                o[bi, :, h] = oh
                lse[bi, h] = lh
        return o, lse

    q, k, v, do = pins.rand_qkv(1, 12, 4, 2, 4, seed=2)
    o_good, _ = orig(q, k, v)
    o_bad, _ = fwd_wrong_group(q, k, v)
    to, _, _, _ = pins.torch_sdpa(q, k, v, do)
    assert np.allclose(o_good, to, rtol=1e-10, atol=1e-11)
    assert not np.allclose(o_bad, to, rtol=1e-10, atol=1e-11)


def test_lse_closed_form_catches_log2(monkeypatch):
    orig = oa.head_forward

    def fwd_log2(qh, kh, vh, scale):
        o, lse, p = orig(qh, kh, vh, scale)
        return o, lse / np.log(2.0) if len(lse) > 1 else lse * 1.5, p

    monkeypatch.setattr(oa, "head_forward", fwd_log2)
    with pytest.raises(AssertionError):
        pins.test_zero_query_prefix_mean()
