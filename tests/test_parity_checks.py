"""The per-row parity check itself (CPU): outputs that differ from the oracle
only by the rounding the kernels do pass; a single stale, zeroed or partly
written row, or a single wrong element, fails it while the whole-tensor norm
still passes."""

import numpy as np
import pytest
import torch

from causal_head_attention_gb300.inputs import make_inputs, small
from tests.parity import TOL, check_rows, full_reference, rel_fro


@pytest.fixture(scope="module")
def case():
    w = small("rowcheck", 2, 4, 2, 300, 64, "bf16", seed=3)
    q, k, v, do = make_inputs(w)
    return full_reference(q, k, v, do)


def bf16_rounded(ref):
    """The reference with every element rounded to bf16 (an output's own rounding)
    and LSE perturbed by 1e-6: what a correct kernel returns at least."""
    out = {}
    for n, a in ref.items():
        if n == "LSE":
            out[n] = a + 1e-6
        else:
            out[n] = torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    return out


def test_rounded_outputs_pass(case):
    check_rows("rounded", bf16_rounded(case), case, "bf16")


@pytest.fixture(scope="module")
def big():
    """Synthetic outputs with 131072 rows per tensor: at this size one bad row
    moves the whole-tensor norm by well under its bound. dQ's first query row
    of every head is exactly zero, as in real attention."""
    g = np.random.default_rng(0)
    o = g.standard_normal((1, 2048, 64, 64))
    dq = g.standard_normal((1, 2048, 64, 64))
    dq[:, 0] = 0.0
    lse = g.standard_normal((1, 64, 2048))
    return {"O": o, "dQ": dq, "LSE": lse}


@pytest.mark.parametrize(
    "name,mutate",
    [
        ("stale row", lambda a: a.__setitem__((0, 200, 1), a[0, 72, 1])),   # a row from another tile
        ("zeroed half row", lambda a: a.__setitem__((0, 150, 3, slice(32, 64)), 0.0)),
        ("one element", lambda a: a.__setitem__((0, 1999, 2, 5), a[0, 1999, 2, 5] + 3.0)),
        ("noise in a zero row", lambda a: a.__setitem__((0, 0, 7), 0.2)),
    ],
)
@pytest.mark.parametrize("out", ["O", "dQ"])
def test_single_bad_row_fails_though_whole_norm_passes(big, name, mutate, out):
    got = bf16_rounded(big)
    check_rows("rounded", got, big, "bf16")
    mutate(got[out])
    assert rel_fro(got[out], big[out]) <= TOL["bf16"][out], "the whole-tensor norm should not see it"
    with pytest.raises(AssertionError, match=out):
        check_rows(name, got, big, "bf16")


def test_bad_key_row_and_lse_fail(case):
    got = bf16_rounded(case)
    got["dV"][1, 10, 0] = got["dV"][1, 11, 0]
    with pytest.raises(AssertionError, match="dV"):
        check_rows("dV", got, case, "bf16")
    got = bf16_rounded(case)
    got["LSE"][0, 2, 17] += 0.01
    with pytest.raises(AssertionError, match="LSE"):
        check_rows("LSE", got, case, "bf16")
