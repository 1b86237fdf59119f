"""Pins for the materialized-path oracle (probabilities returned, VJP through
both outputs), and mistakes planted in it (on the CPU).

The probabilities and the VJP are checked against code that shares nothing with
the oracle: torch's fp64 softmax of the masked scores, torch autograd of the
loss <dO, O> + <dP, P>, and central finite differences of that loss. Two
invariants of the softmax VJP are checked too: entries of dP above the diagonal
(where P is 0) change nothing, and neither does a constant added to a row's
kept entries (softmax is shift invariant).
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import materialized as om


def rand(b, t, hq, hkv, dh, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((b, t, hq, dh))
    k = rng.standard_normal((b, t, hkv, dh))
    v = rng.standard_normal((b, t, hkv, dh))
    do = rng.standard_normal((b, t, hq, dh))
    dp = rng.standard_normal((b, hq, t, t))
    return q, k, v, do, dp


def torch_path(q, k, v):
    """fp64 torch: scores, masked softmax, context; heads on dim 1."""
    hq, hkv = q.shape[2], k.shape[2]
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = kt.repeat_interleave(hq // hkv, dim=2)
    vv = vt.repeat_interleave(hq // hkv, dim=2)
    t = q.shape[1]
    s = torch.einsum("bihd,bjhd->bhij", qt, kk) / np.sqrt(q.shape[3])
    mask = torch.ones(t, t, dtype=torch.bool).tril()
    p = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, vv)
    return qt, kt, vt, p, o


@pytest.mark.parametrize("shape", [(2, 7, 2, 2, 4), (1, 9, 4, 2, 8), (1, 1, 2, 1, 4)])
def test_probs_match_torch_softmax(shape):
    q, k, v, _, _ = rand(*shape, seed=1)
    o, p, lse = oracle.attention_probs(q, k, v)
    _, _, _, tp, to = torch_path(q, k, v)
    assert np.allclose(p, tp.detach().numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    t = shape[1]
    assert np.all(p[..., np.triu_indices(t, 1)[0], np.triu_indices(t, 1)[1]] == 0)


@pytest.mark.parametrize("shape", [(2, 6, 2, 2, 4), (1, 8, 4, 2, 4)])
def test_vjp_matches_torch_autograd(shape):
    q, k, v, do, dp = rand(*shape, seed=2)
    dq, dk, dv = oracle.materialized_backward(q, k, v, do, dp)
    qt, kt, vt, tp, to = torch_path(q, k, v)
    loss = (to * torch.tensor(do)).sum() + (tp * torch.tensor(dp)).sum()
    loss.backward()
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_vjp_finite_differences():
    q, k, v, do, dp = rand(1, 5, 2, 1, 3, seed=3)

    def loss(q_, k_, v_):
        o, p, _ = oracle.attention_probs(q_, k_, v_)
        return float(np.sum(o * do) + np.sum(p * dp))

    dq, dk, dv = oracle.materialized_backward(q, k, v, do, dp)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = x.copy(); xp[i] += eps
            xm = x.copy(); xm[i] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[i]) < 1e-6 * (1 + abs(fd)), (i, fd, g[i])


def test_no_probability_gradient_equals_full_sequence_backward():
    q, k, v, do, _ = rand(2, 9, 4, 2, 8, seed=4)
    a = oracle.materialized_backward(q, k, v, do, None)
    b = oracle.attention_backward(q, k, v, do)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-11, atol=1e-13)


def test_vjp_invariances():
    q, k, v, do, dp = rand(1, 8, 2, 2, 4, seed=5)
    base = oracle.materialized_backward(q, k, v, do, dp)
    t = q.shape[1]
    above = np.triu(np.ones((t, t), dtype=bool), 1)
    dp2 = dp.copy()
    dp2[..., above] = 1e3 * np.random.default_rng(6).standard_normal(dp2[..., above].shape)
    shift = np.random.default_rng(7).standard_normal((1, 2, t, 1))
    dp2 = dp2 + np.where(above, 0.0, shift)
    got = oracle.materialized_backward(q, k, v, do, dp2)
    for x, y in zip(got, base):
        assert np.allclose(x, y, rtol=1e-9, atol=1e-11)


def test_causal_softmax_matches_torch_and_head_forward():
    rng = np.random.default_rng(11)
    s = rng.standard_normal((3, 9, 9)) * 4
    p, lse = oracle.causal_softmax(s, 0.7)
    mask = torch.ones(9, 9, dtype=torch.bool).tril()
    st = torch.tensor(s, dtype=torch.float64, requires_grad=True)
    tp = torch.softmax((0.7 * st).masked_fill(~mask, float("-inf")), dim=-1)
    assert np.allclose(p, tp.detach().numpy(), rtol=1e-12, atol=1e-15)
    assert np.allclose(lse, torch.logsumexp((0.7 * st).masked_fill(~mask, float("-inf")), -1).detach().numpy())
    g = rng.standard_normal((3, 9, 9))
    (tp * torch.tensor(g)).sum().backward()
    assert np.allclose(oracle.causal_softmax_vjp(p, g, 0.7), st.grad.numpy(), rtol=1e-11, atol=1e-13)
    q, k, v, _, _ = rand(1, 9, 1, 1, 4, seed=12)
    _, _, ph = oracle.head_forward(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.5)
    p2, _ = oracle.causal_softmax(q[0, :, 0] @ k[0, :, 0].T, 0.5)
    assert np.allclose(p2, ph, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _bwd_no_rowsum(qh, kh, vh, doh, dph, p, scale):
    dp = oracle.contract(doh, np.asarray(vh).T) + (0 if dph is None else dph)
    ds = p * dp  # dropped the rowsum term
    return scale * oracle.contract(ds, kh), scale * oracle.contract(ds.T, qh), oracle.contract(p.T, doh)


_ORIG = om.head_backward_probs


def _bwd_dp_up_ignored(qh, kh, vh, doh, dph, p, scale):
    return _ORIG(qh, kh, vh, doh, None, p, scale)


def _bwd_dp_up_transposed(qh, kh, vh, doh, dph, p, scale):
    return _ORIG(qh, kh, vh, doh, None if dph is None else dph.T, p, scale)


@pytest.mark.parametrize("mutant", [_bwd_no_rowsum, _bwd_dp_up_ignored, _bwd_dp_up_transposed])
def test_pins_catch_mutants(monkeypatch, mutant):
    monkeypatch.setattr(om, "head_backward_probs", mutant)
    with pytest.raises(AssertionError):
        test_vjp_matches_torch_autograd((1, 8, 4, 2, 4))
