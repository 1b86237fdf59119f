"""Pins for the paged-decode oracle, and mistakes planted in it (on the CPU).

Paged decode ("Execution Backends and the Python ABI", "Incremental attention")
is one query token per request attending over its cached keys and values, each
fetched through the request's page table. The pins tie it to facts outside its
own code:

* a contiguous cache (page table 0, 1, 2, ...) gives, for a request of length
  L, exactly row L - 1 of the full-sequence causal attention over the first L
  positions (the full-sequence oracle is pinned against torch, closed forms and
  finite differences in test_oracle_pins.py); checked with grouped-query heads
  and lengths that end inside a page, on a page boundary and at one position;
* scattering the same logical cache to other physical pages (a permuted table)
  changes nothing: every output is bit-identical;
* whatever sits in the pool past a request's length, or in table entries past
  its last page, changes nothing;
* L = 1 has the closed form O = V[0], LSE = scale * q . k[0];
* equal keys give the mean of the values, LSE = s + ln L.

The second half plants plausible mistakes (table ignored, page and offset
swapped, interleaved head groups, one position too many, the scale dropped)
and shows that a pin fails for each.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import decode as pd


def contiguous_pools(k, v, page_size):
    """[B,T,Hkv,Dh] caches -> pools [B*npg, Hkv, page_size, Dh] with request b on
    pages b*npg .. b*npg+npg-1 in order, and the matching page table."""
    B, T, Hkv, Dh = k.shape
    npg = -(-T // page_size)
    pad = npg * page_size - T
    kp = np.pad(k, ((0, 0), (0, pad), (0, 0), (0, 0)), constant_values=7.0)
    vp = np.pad(v, ((0, 0), (0, pad), (0, 0), (0, 0)), constant_values=-7.0)
    kp = kp.reshape(B, npg, page_size, Hkv, Dh).transpose(0, 1, 3, 2, 4).reshape(B * npg, Hkv, page_size, Dh)
    vp = vp.reshape(B, npg, page_size, Hkv, Dh).transpose(0, 1, 3, 2, 4).reshape(B * npg, Hkv, page_size, Dh)
    table = np.arange(B * npg, dtype=np.int64).reshape(B, npg)
    return kp, vp, table


def rand_cache(B, T, Hq, Hkv, Dh, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, Dh))
    k = rng.standard_normal((B, T, Hkv, Dh))
    v = rng.standard_normal((B, T, Hkv, Dh))
    return q, k, v


@pytest.mark.parametrize("page_size", [1, 4, 8])
def test_contiguous_cache_equals_causal_row(page_size):
    B, T, Hq, Hkv, Dh = 2, 19, 4, 2, 8
    q, k, v = rand_cache(B, T, Hq, Hkv, Dh, seed=page_size)
    o_full, lse_full = oracle.attention_forward(q, k, v)
    kp, vp, table = contiguous_pools(k, v, page_size)
    for L in (1, page_size, page_size + 1, 2 * page_size, T):
        if L > T:
            continue
        seq = np.array([L, max(1, L - 1)])
        o, lse = oracle.paged_decode(q[np.arange(B), seq - 1], kp, vp, table, seq)
        for b in range(B):
            assert np.allclose(o[b], o_full[b, seq[b] - 1], rtol=1e-12, atol=1e-13), (L, b)
            assert np.allclose(lse[b], lse_full[b, :, seq[b] - 1], rtol=1e-12, atol=1e-13), (L, b)


def test_page_permutation_invariance():
    B, T, Hq, Hkv, Dh, ps = 3, 23, 2, 2, 4, 4
    q, k, v = rand_cache(B, T, Hq, Hkv, Dh, seed=5)
    kp, vp, table = contiguous_pools(k, v, ps)
    seq = np.array([23, 9, 16])
    q1 = q[:, 0]
    o0, lse0 = oracle.paged_decode(q1, kp, vp, table, seq)
    rng = np.random.default_rng(6)
    P = kp.shape[0]
    perm = rng.permutation(P + 5)[:P]  # new physical slot of each old page, in a larger pool
    kq = rng.standard_normal((P + 5,) + kp.shape[1:])
    vq = rng.standard_normal((P + 5,) + vp.shape[1:])
    kq[perm] = kp
    vq[perm] = vp
    o1, lse1 = oracle.paged_decode(q1, kq, vq, perm[table], seq)
    assert np.array_equal(o0, o1)
    assert np.array_equal(lse0, lse1)


def test_tail_and_unused_entries_ignored():
    B, T, Hq, Hkv, Dh, ps = 2, 13, 2, 1, 4, 4
    q, k, v = rand_cache(B, T, Hq, Hkv, Dh, seed=7)
    kp, vp, table = contiguous_pools(k, v, ps)
    seq = np.array([6, 13])
    o0, lse0 = oracle.paged_decode(q[:, 0], kp, vp, table, seq)
    kp2, vp2, table2 = kp.copy(), vp.copy(), table.copy()
    # request 0 uses pages 0 and 1 up to offset 1: poison the rest of page 1 and pages 2, 3
    kp2[1, :, 2:] = 1e6
    vp2[1, :, 2:] = np.nan
    table2[0, 2:] = -1
    o1, lse1 = oracle.paged_decode(q[:, 0], kp2, vp2, table2, seq)
    assert np.array_equal(o0, o1)
    assert np.array_equal(lse0, lse1)


def test_single_position_closed_form():
    rng = np.random.default_rng(8)
    Hq, Hkv, Dh, ps = 4, 2, 16, 8
    q = rng.standard_normal((1, Hq, Dh))
    kp = rng.standard_normal((3, Hkv, ps, Dh))
    vp = rng.standard_normal((3, Hkv, ps, Dh))
    table = np.array([[2, 0]])
    o, lse = oracle.paged_decode(q, kp, vp, table, np.array([1]))
    for h in range(Hq):
        kv = h // 2
        assert np.allclose(o[0, h], vp[2, kv, 0], rtol=0, atol=1e-15)
        assert math.isclose(lse[0, h], float(q[0, h] @ kp[2, kv, 0]) / math.sqrt(Dh), rel_tol=1e-13)


def test_equal_keys_give_value_mean():
    rng = np.random.default_rng(9)
    Hq, Hkv, Dh, ps, L = 2, 2, 8, 4, 11
    q = rng.standard_normal((1, Hq, Dh))
    kp = np.broadcast_to(rng.standard_normal((1, Hkv, 1, Dh)), (3, Hkv, ps, Dh)).copy()
    vp = rng.standard_normal((3, Hkv, ps, Dh))
    table = np.array([[1, 2, 0]])
    o, lse = oracle.paged_decode(q, kp, vp, table, np.array([L]))
    vals = np.concatenate([vp[1].transpose(1, 0, 2), vp[2].transpose(1, 0, 2), vp[0].transpose(1, 0, 2)])[:L]
    for h in range(Hq):
        s = float(q[0, h] @ kp[0, h, 0]) / math.sqrt(Dh)
        assert np.allclose(o[0, h], vals[:, h].mean(axis=0), rtol=1e-12, atol=1e-14)
        assert math.isclose(lse[0, h], s + math.log(L), rel_tol=1e-12)


def test_rejects_empty_request_and_bad_groups():
    q = np.zeros((1, 3, 4))
    kp = np.zeros((1, 2, 4, 4))
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kp, kp, np.array([[0]]), np.array([1]))
    q = np.zeros((1, 2, 4))
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kp, kp, np.array([[0]]), np.array([0]))


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _gather_ignoring_table(pool, table_row, length):
    ps = pool.shape[2]
    return np.stack([pool[t // ps, :, t % ps, :] for t in range(length)]).astype(np.float64)


def _gather_swapped(pool, table_row, length):
    ps = pool.shape[2]
    rows = []
    for t in range(length):
        page, off = t % ps, t // ps
        rows.append(pool[int(table_row[min(page, len(table_row) - 1)]), :, min(off, ps - 1), :])
    return np.stack(rows).astype(np.float64)


def _gather_one_too_many(pool, table_row, length):
    ps = pool.shape[2]
    n = min(length + 1, len(table_row) * ps)
    return np.stack([pool[int(table_row[t // ps]), :, t % ps, :] for t in range(n)]).astype(np.float64)


def _run_pins():
    test_contiguous_cache_equals_causal_row(4)
    test_page_permutation_invariance()
    test_tail_and_unused_entries_ignored()
    test_single_position_closed_form()
    test_equal_keys_give_value_mean()


@pytest.mark.parametrize("mutant", [_gather_ignoring_table, _gather_swapped, _gather_one_too_many])
def test_pins_catch_gather_mutants(monkeypatch, mutant):
    monkeypatch.setattr(pd, "gather_positions", mutant)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_interleaved_groups(monkeypatch):
    monkeypatch.setattr(pd, "kv_head", lambda h, g: h % 2)
    with pytest.raises(AssertionError):
        _run_pins()


def test_pins_catch_missing_scale(monkeypatch):
    monkeypatch.setattr(pd, "default_scale", lambda dh: 1.0)
    with pytest.raises(AssertionError):
        _run_pins()
