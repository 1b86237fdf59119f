"""Pins for the padded / variable-length oracle, and mistakes planted in it.

L_b = T reduces to the (separately pinned) full-sequence oracle; nothing at a
padding position (inputs or upstream gradient) may reach an output at a real
position; padding outputs are exactly zero (LSE -inf); an all-padding
sequence gives zeros, not NaN (the fully-masked-row guard); central finite
differences of <dO, O> over real positions.
"""

import numpy as np
import pytest

import oracle


def rand(b, t, hq, hkv, dh, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((b, t, hq, dh)), rng.standard_normal((b, t, hkv, dh)),
            rng.standard_normal((b, t, hkv, dh)), rng.standard_normal((b, t, hq, dh)))


def test_full_length_is_full_sequence():
    q, k, v, do = rand(2, 9, 4, 2, 4, 1)
    lens = [9, 9]
    o, lse = oracle.attention_forward_varlen(q, k, v, lens)
    o2, lse2 = oracle.attention_forward(q, k, v)
    assert np.allclose(o, o2, rtol=1e-13, atol=1e-14) and np.allclose(lse, lse2, rtol=1e-13)
    for a, b in zip(oracle.attention_backward_varlen(q, k, v, do, lens), oracle.attention_backward(q, k, v, do)):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


def test_padding_never_reaches_real_positions():
    q, k, v, do = rand(3, 10, 2, 1, 4, 2)
    lens = np.array([10, 4, 0])
    base_f = oracle.attention_forward_varlen(q, k, v, lens)
    base_b = oracle.attention_backward_varlen(q, k, v, do, lens)
    rng = np.random.default_rng(3)
    q2, k2, v2, do2 = (x.copy() for x in (q, k, v, do))
    for bi, n in enumerate(lens):
        for x in (q2, k2, v2, do2):
            x[bi, n:] = 1e3 * rng.standard_normal(x[bi, n:].shape)
    f2 = oracle.attention_forward_varlen(q2, k2, v2, lens)
    b2 = oracle.attention_backward_varlen(q2, k2, v2, do2, lens)
    for a, b in zip(base_f + base_b, f2 + b2):
        assert np.array_equal(a, b)


def test_padding_outputs_zero_and_empty_sequence_guard():
    q, k, v, do = rand(2, 6, 2, 2, 4, 4)
    lens = [3, 0]
    o, lse = oracle.attention_forward_varlen(q, k, v, lens)
    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, lens)
    assert np.all(o[0, 3:] == 0) and np.all(o[1] == 0)
    assert np.all(np.isneginf(lse[0, :, 3:])) and np.all(np.isneginf(lse[1]))
    for g in (dq, dk, dv):
        assert np.all(g[0, 3:] == 0) and np.all(g[1] == 0) and np.all(np.isfinite(g))
    assert np.all(np.isfinite(o))


def test_finite_differences_real_positions():
    q, k, v, do = rand(2, 5, 2, 1, 3, 5)
    lens = [5, 3]

    def loss(q_, k_, v_):
        o, _ = oracle.attention_forward_varlen(q_, k_, v_, lens)
        return float(np.sum(o * do * (np.arange(5)[None, :, None, None] < np.array(lens)[:, None, None, None])))

    dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, lens)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = x.copy(); xp[i] += eps
            xm = x.copy(); xm[i] -= eps
            ap = [xp if y is x else y for y in (q, k, v)]
            am = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*ap) - loss(*am)) / (2 * eps)
            assert abs(fd - g[i]) < 1e-6 * (1 + abs(fd)), (i, fd, g[i])


def test_rejects_bad_lengths():
    q, k, v, _ = rand(2, 4, 1, 1, 2, 6)
    with pytest.raises(ValueError):
        oracle.attention_forward_varlen(q, k, v, [5, 1])
    with pytest.raises(ValueError):
        oracle.attention_forward_varlen(q, k, v, [-1, 1])


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _fwd_padding_rows_kept(q, k, v, lens, scale=None):
    return oracle.attention_forward(q, k, v, scale)  # padding rows not zeroed, no guard


def _bwd_padding_dout_used(q, k, v, do, lens, scale=None):
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale)  # gradients from padding queries
    for bi, n in enumerate(lens):
        dq[bi, n:] = 0
    return dq, dk, dv


def test_pins_catch_forward_mutant(monkeypatch):
    monkeypatch.setattr(oracle, "attention_forward_varlen", _fwd_padding_rows_kept)
    with pytest.raises(AssertionError):
        test_padding_outputs_zero_and_empty_sequence_guard()


def test_pins_catch_backward_mutant(monkeypatch):
    monkeypatch.setattr(oracle, "attention_backward_varlen", _bwd_padding_dout_used)
    with pytest.raises(AssertionError):
        test_padding_never_reaches_real_positions()
