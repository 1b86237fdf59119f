"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

Each check below would fail on a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong mask or head map);
tests/test_oracle_mutations.py plants such mistakes and shows that they do.
No GPU is needed.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_qkv(b, t, hq, hkv, dh, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((b, t, hq, dh)) * scale
    k = rng.standard_normal((b, t, hkv, dh)) * scale
    v = rng.standard_normal((b, t, hkv, dh))
    do = rng.standard_normal((b, t, hq, dh))
    return q, k, v, do


def read_golden(name):
    blocks, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head = line.split()
            if head[0].isalpha():
                cur = head[0]
                blocks[cur] = {"dims": [int(x) for x in head[1:]], "vals": []}
            else:
                blocks[cur]["vals"].extend(float(x) for x in head)
    return blocks


# --- worked example from the pages -------------------------------------------------

def test_contraction_worked_example():
    g = read_golden("matmul_worked_example.txt")
    a = np.array(g["left"]["vals"]).reshape(g["left"]["dims"])
    b = np.array(g["right"]["vals"]).reshape(g["right"]["dims"])
    want = np.array(g["product"]["vals"]).reshape(g["product"]["dims"])
    got = oracle.contract(a, b)
    assert got.shape == tuple(g["product"]["dims"])
    assert np.array_equal(got, want)


def test_large_logits_stay_finite():
    """A query/key pair whose causal scores in the last row are exactly the
    page's [10000, 10001, 10002] example (Dh=1 so the scale is 1)."""
    g = read_golden("stable_softmax_large_logits.txt")
    z = np.array(g["logits"]["vals"])
    t = z.size
    q = np.ones((t, 1))
    k = z.reshape(t, 1)
    v = np.eye(t)[:, :1] * 0 + np.arange(t, dtype=np.float64).reshape(t, 1)
    o, lse, p = oa.head_forward(q, k, v, 1.0)
    assert np.all(np.isfinite(p)) and np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    shifted = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    closed = np.exp(np.arange(t)) / np.exp(np.arange(t)).sum()  # softmax([0,1,2])
    assert np.allclose(shifted, closed, rtol=0, atol=1e-15)
    assert np.allclose(p[-1], closed, rtol=1e-13, atol=1e-15)
    assert abs(lse[-1] - (z.max() + math.log(np.exp(z - z.max()).sum()))) < 1e-9


def test_empty_row_rejected():
    with pytest.raises(ValueError):
        oa.head_forward(np.zeros((0, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 0.5)


# --- invariants ---------------------------------------------------------------------

def test_rows_sum_to_one_and_mask():
    q, k, v, _ = rand_qkv(1, 37, 1, 1, 8, seed=1, scale=2.0)
    _, _, p = oa.head_forward(q[0, :, 0], k[0, :, 0], v[0, :, 0], oracle.default_scale(8))
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p[np.triu_indices(37, 1)] == 0.0)
    assert np.all(p[np.tril_indices(37)] > 0.0)
    assert p[0, 0] == 1.0


def test_single_position_closed_form():
    """T=1: the only key is the query's own, so O = V and LSE = scale*q.k."""
    q, k, v, do = rand_qkv(2, 1, 4, 2, 8, seed=2)
    s = oracle.default_scale(8)
    o, lse = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    g = 2
    for h in range(4):
        assert np.allclose(o[:, 0, h], v[:, 0, h // g], rtol=0, atol=1e-15)
        assert np.allclose(lse[:, h, 0], s * np.sum(q[:, 0, h] * k[:, 0, h // g], axis=-1), atol=1e-14)
    assert np.allclose(dq, 0, atol=1e-15) and np.allclose(dk, 0, atol=1e-15)
    want_dv = do.reshape(2, 1, 2, g, 8).sum(axis=3)
    assert np.allclose(dv, want_dv, atol=1e-14)


def test_zero_query_prefix_mean():
    """Q=0: all allowed scores are 0, so O[t] is the mean of V[0..t] and LSE[t]=ln(t+1)."""
    q, k, v, do = rand_qkv(1, 19, 2, 1, 4, seed=3)
    q[:] = 0.0
    o, lse = oracle.attention_forward(q, k, v)
    _, dk, _ = oracle.attention_backward(q, k, v, do)
    csum = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, 20)[:, None]
    for h in range(2):
        assert np.allclose(o[0, :, h], csum, atol=1e-14)
        assert np.allclose(lse[0, h], np.log(np.arange(1, 20)), atol=1e-14)
    assert np.allclose(dk, 0, atol=1e-14)


def test_zero_key_prefix_mean():
    q, k, v, _ = rand_qkv(1, 11, 1, 1, 4, seed=4)
    k[:] = 0.0
    o, lse = oracle.attention_forward(q, k, v)
    csum = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, 12)[:, None]
    assert np.allclose(o[0, :, 0], csum, atol=1e-14)
    assert np.allclose(lse[0, 0], np.log(np.arange(1, 12)), atol=1e-14)


def test_causality_future_perturbation():
    """Changing K/V at positions > t leaves O, LSE and dQ at positions <= t unchanged."""
    q, k, v, do = rand_qkv(1, 24, 2, 2, 8, seed=5)
    t = 9
    o1, l1 = oracle.attention_forward(q, k, v)
    dq1, _, _ = oracle.attention_backward(q, k, v, do)
    k2, v2 = k.copy(), v.copy()
    rng = np.random.default_rng(99)
    k2[:, t + 1:] += rng.standard_normal(k2[:, t + 1:].shape) * 5
    v2[:, t + 1:] += rng.standard_normal(v2[:, t + 1:].shape) * 5
    o2, l2 = oracle.attention_forward(q, k2, v2)
    dq2, _, _ = oracle.attention_backward(q, k2, v2, do)
    assert np.array_equal(o1[:, : t + 1], o2[:, : t + 1])
    assert np.array_equal(l1[:, :, : t + 1], l2[:, :, : t + 1])
    assert np.array_equal(dq1[:, : t + 1], dq2[:, : t + 1])
    assert not np.allclose(o1[:, t + 1:], o2[:, t + 1:])


def test_key_shift_invariance():
    """Adding c to every key shifts each score row by scale*q_i.c: O is unchanged
    and LSE_i moves by exactly that amount."""
    q, k, v, _ = rand_qkv(1, 16, 2, 1, 8, seed=6)
    c = np.random.default_rng(7).standard_normal(8)
    s = oracle.default_scale(8)
    o1, l1 = oracle.attention_forward(q, k, v)
    o2, l2 = oracle.attention_forward(q, k + c, v)
    assert np.allclose(o1, o2, atol=1e-12)
    shift = s * np.einsum("bthd,d->bht", q, c)
    assert np.allclose(l2 - l1, shift, atol=1e-12)


def test_d_identity():
    """D_i = sum_d dO*O equals sum_j P*dP (the identity the backward relies on)."""
    q, k, v, do = rand_qkv(1, 21, 1, 1, 6, seed=8)
    s = oracle.default_scale(6)
    qh, kh, vh, doh = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    o, _, p = oa.head_forward(qh, kh, vh, s)
    _, _, _, d = oa.head_backward(qh, kh, vh, o, doh, p, s)
    dp = doh @ vh.T
    assert np.allclose(d, np.sum(p * dp, axis=1), atol=1e-12)


# --- brute force: central finite differences -----------------------------------------

def fd_check(b, t, hq, hkv, dh, seed, h=1e-6, rtol=2e-6):
    q, k, v, do = rand_qkv(b, t, hq, hkv, dh, seed=seed)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_forward(q_, k_, v_)
        return float(np.sum(do * o))

    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k, v)
            x[idx] = old - h
            lm = loss(q, k, v)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < rtol, f"finite-difference mismatch {err:.3e}"


def test_finite_differences_gqa():
    fd_check(1, 5, 2, 1, 4, seed=10)


def test_finite_differences_mha():
    fd_check(2, 4, 2, 2, 3, seed=11)


# --- an independent second algorithm: tile-8 online softmax ------------------------------

def flash_tile8_forward(qh, kh, vh, scale, tile=8):
    """Online-softmax forward over 8-key tiles (the pages' CPU Flash design idea),
    written independently of the oracle: running max m, running sum l, O rescaled."""
    t, dh = qh.shape
    o = np.zeros((t, vh.shape[1]))
    lse = np.zeros(t)
    for i0 in range(0, t, tile):
        rows = range(i0, min(i0 + tile, t))
        for i in rows:
            m, l = -np.inf, 0.0
            acc = np.zeros(vh.shape[1])
            for j0 in range(0, i + 1, tile):
                js = np.arange(j0, min(j0 + tile, i + 1))
                sc = np.array([scale * float(np.dot(qh[i], kh[j])) for j in js])
                m_new = max(m, sc.max())
                alpha = math.exp(m - m_new) if m != -np.inf else 0.0
                e = np.exp(sc - m_new)
                l = l * alpha + e.sum()
                acc = acc * alpha + e @ vh[js]
                m = m_new
            o[i] = acc / l
            lse[i] = m + math.log(l)
    return o, lse


def flash_tile8_backward(qh, kh, vh, oh, doh, lse, scale, tile=8):
    """Recompute-from-LSE backward over 8x8 tiles (key tile outer, query tile inner)."""
    t, dh = qh.shape
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    dd = np.array([float(np.dot(doh[i], oh[i])) for i in range(t)])
    for j0 in range(0, t, tile):
        js = np.arange(j0, min(j0 + tile, t))
        for i0 in range(j0 - j0 % tile, t, tile):
            for i in range(max(i0, j0), min(i0 + tile, t)):
                for j in js:
                    if j > i:
                        continue
                    p = math.exp(scale * float(np.dot(qh[i], kh[j])) - lse[i])
                    dv[j] += p * doh[i]
                    dp = float(np.dot(doh[i], vh[j]))
                    ds = p * (dp - dd[i])
                    dq[i] += scale * ds * kh[j]
                    dk[j] += scale * ds * qh[i]
    return dq, dk, dv


def test_tile8_flash_matches_oracle():
    q, k, v, do = rand_qkv(1, 29, 2, 1, 5, seed=12, scale=1.5)
    s = oracle.default_scale(5)
    o, lse = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    dk2 = np.zeros_like(dk)
    dv2 = np.zeros_like(dv)
    for h in range(2):
        of, lf = flash_tile8_forward(q[0, :, h], k[0, :, 0], v[0, :, 0], s)
        assert np.allclose(of, o[0, :, h], rtol=0, atol=1e-12)
        assert np.allclose(lf, lse[0, h], rtol=0, atol=1e-12)
        dqf, dkf, dvf = flash_tile8_backward(q[0, :, h], k[0, :, 0], v[0, :, 0], of, do[0, :, h], lf, s)
        assert np.allclose(dqf, dq[0, :, h], atol=1e-12)
        dk2[0, :, 0] += dkf
        dv2[0, :, 0] += dvf
    assert np.allclose(dk2, dk, atol=1e-12)
    assert np.allclose(dv2, dv, atol=1e-12)


# --- library routine: torch fp64 scaled_dot_product_attention ---------------------------

def torch_sdpa(q, k, v, do):
    g = q.shape[2] // k.shape[2]
    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_(True)
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_(True)
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_(True)
    kk = tk.repeat_interleave(g, dim=1)
    vv = tv.repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=True)
    o.backward(torch.tensor(do).permute(0, 2, 1, 3))
    perm = lambda x: x.permute(0, 2, 1, 3).detach().numpy()  # noqa: E731
    return perm(o), perm(tq.grad), perm(tk.grad), perm(tv.grad)


@pytest.mark.parametrize("shape", [(2, 64, 4, 4, 16), (1, 33, 4, 2, 8), (1, 70, 6, 2, 32)])
def test_matches_torch_sdpa_fp64(shape):
    q, k, v, do = rand_qkv(*shape, seed=13)
    o, _ = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    to, tdq, tdk, tdv = torch_sdpa(q, k, v, do)
    for a, b in ((o, to), (dq, tdq), (dk, tdk), (dv, tdv)):
        assert np.allclose(a, b, rtol=1e-10, atol=1e-11)


def test_group_reference_matches_whole_tensor():
    q, k, v, do = rand_qkv(2, 20, 6, 2, 8, seed=14)
    o, lse = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    for b in range(2):
        for kv in range(2):
            r = oracle.group_reference(q, k, v, do, b, kv)
            hs = slice(kv * 3, kv * 3 + 3)
            assert np.allclose(r["O"], o[b, :, hs], atol=1e-14)
            assert np.allclose(r["LSE"], lse[b, hs], atol=1e-14)
            assert np.allclose(r["dQ"], dq[b, :, hs], atol=1e-14)
            assert np.allclose(r["dK"], dk[b, :, kv], atol=1e-14)
            assert np.allclose(r["dV"], dv[b, :, kv], atol=1e-14)


def test_backward_of_a_given_output():
    """The backward handed an output o reads it only through D = rowsum(dO * o).
    With the exact output it is the exact VJP; with o = O + E every row's D
    moves by delta_i = sum_d dO[i,d] E[i,d], so dS loses P[i,j] delta_i: dQ
    moves by -scale * delta_i * (P K)_i, dK by -scale * sum_i P[i,j] delta_i
    Q_i, and dV not at all."""
    q, k, v, do = rand_qkv(2, 17, 4, 2, 8, seed=16)
    o, _ = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    same = oracle.attention_backward(q, k, v, do, o=o)
    for a, b in zip(same, (dq, dk, dv)):
        assert np.allclose(a, b, atol=1e-14)
    e = np.random.default_rng(17).standard_normal(o.shape) * 1e-2
    dq2, dk2, dv2 = oracle.attention_backward(q, k, v, do, o=o + e)
    sc = oracle.default_scale(8)
    assert np.allclose(dv2, dv, atol=1e-14)
    for b in range(2):
        for h in range(4):
            kv = h // 2
            _, _, p = oa.head_forward(q[b, :, h], k[b, :, kv], v[b, :, kv], sc)
            delta = np.sum(do[b, :, h] * e[b, :, h], axis=1)
            assert np.allclose(dq2[b, :, h] - dq[b, :, h], -sc * delta[:, None] * (p @ k[b, :, kv]), atol=1e-12)
    for b in range(2):
        for kv in range(2):
            want = np.zeros((17, 8))
            for h in (2 * kv, 2 * kv + 1):
                _, _, p = oa.head_forward(q[b, :, h], k[b, :, kv], v[b, :, kv], sc)
                delta = np.sum(do[b, :, h] * e[b, :, h], axis=1)
                want += -sc * (p * delta[:, None]).T @ q[b, :, h]
            assert np.allclose(dk2[b, :, kv] - dk[b, :, kv], want, atol=1e-12)
    r = oracle.group_reference(q, k, v, do, 1, 1, o=o + e)
    assert np.allclose(r["given_o"]["dQ"], dq2[1, :, 2:4], atol=1e-14)
    assert np.allclose(r["given_o"]["dK"], dk2[1, :, 1], atol=1e-14)
    assert np.allclose(r["dQ"], dq[1, :, 2:4], atol=1e-14)


def test_gqa_divisibility_rejected():
    q, k, v, _ = rand_qkv(1, 4, 3, 2, 4, seed=15)
    with pytest.raises(ValueError):
        oracle.attention_forward(q, k, v)
