"""Pin of the oracle's routed combine with distinct experts ("Speculating on a
Strix Halo", section "What the pieces cost": each token's output is the
weighted sum of its own top-K experts' outputs, the weights being the softmax
of the router logits over the selected experts).

The layer is built so that every quantity has a closed form: expert e's
output is a multiple of the unit vector e (a different coordinate per
expert), its size set by its own up weight, and the router logits of a row
are fixed multiples of ln 4 and ln 2.  A weight paired with the wrong slot, a
row's weights taken from another row, or a slot's expert output taken from
another slot each put a wrong number in some coordinate; the planted-mistake
test below compiles those three mistakes into copies of the oracle and shows
that each one fails the closed form.  CPU only."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from tests import _mutants

LN2, LN3, LN4 = (float(np.float32(math.log(v))) for v in (2.0, 3.0, 4.0))  # as stored (fp32)
C_UP = (1.0, 2.0, 3.0)  # up weight of expert e: sets the size of its output


def _layer(norm_topk: int) -> oracle.Layer:
    d, I, E, K = 4, 1, 3, 2
    wr = np.zeros((E, d), dtype=np.float32)
    wr[:, 0] = [LN4, 0.0, -LN2]
    wg = np.zeros((E, I, d), dtype=np.float32)
    wg[:, 0, 1] = LN3
    wu = np.zeros((E, I, d), dtype=np.float32)
    wu[:, 0, 1] = C_UP
    wd = np.zeros((E, d, I), dtype=np.float32)
    for e in range(E):
        wd[e, e, 0] = 1.0
    return oracle.Layer(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype=oracle.F32, r_dtype=oracle.F32,
                        w_router=wr, w_gate=wg, w_up=wu, w_down=wd, norm_topk=norm_topk)


# rows: x = (s, 1, 0, 0), so row t's logits are s * (ln 4, 0, -ln 2)
X = np.array([[1.0, 1.0, 0.0, 0.0], [-1.0, 1.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]], dtype=np.float32)


def _closed_form(norm_topk: int) -> np.ndarray:
    g = LN3  # gate pre-activation of every expert: ln 3 * x[1]
    h = [g / (1.0 + math.exp(-g)) * c for c in C_UP]  # silu(g) * u, expert e
    out = np.zeros((3, 4))
    for t, s in enumerate(X[:, 0]):
        lg = [s * LN4, 0.0, -s * LN2]
        # top-2 by descending logit, equal logits to the lower expert id
        sel = sorted(range(3), key=lambda e: (-lg[e], e))[:2]
        z = [math.exp(v) for v in lg]
        den = sum(z[e] for e in sel) if norm_topk else sum(z)
        for e in sel:
            out[t, e] += z[e] / den * h[e]
    return out


def test_closed_form_selects_the_expected_experts():
    # row 0 picks experts (0, 1) with weights (4/5, 1/5), row 1 picks (2, 1)
    # with (2/3, 1/3), row 2 has three equal logits and picks (0, 1), 1/2 each
    _, idx, w = oracle.route(_layer(1), X)
    assert idx.tolist() == [[0, 1], [2, 1], [0, 1]]
    assert w[0] == pytest.approx([0.8, 0.2], rel=1e-7)
    assert w[1] == pytest.approx([2.0 / 3.0, 1.0 / 3.0], rel=1e-7)
    assert w[2].tolist() == [0.5, 0.5]


@pytest.mark.parametrize("norm_topk", [1, 0])
def test_routed_combine_equals_closed_form_with_distinct_experts(norm_topk):
    got = oracle.moe_forward(_layer(norm_topk), X)
    want = _closed_form(norm_topk)
    assert np.all(got[:, 3] == 0.0)
    assert got[1, 0] == 0.0 and got[0, 2] == 0.0 and got[2, 2] == 0.0
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0.0)


# Each mistake is a one-fragment edit of oracle.c's combine loop.
MUTANTS = {
    "weight of the mirrored slot": ("w[t * K + s] * y[j]", "w[t * K + (K - 1 - s)] * y[j]"),
    "weights of the next row": ("w[t * K + s] * y[j]", "w[((t + 1) % k) * K + s] * y[j]"),
    "expert output of the mirrored slot": ("ys + (size_t)(t * K + s) * d", "ys + (size_t)(t * K + (K - 1 - s)) * d"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_pairing_mistakes_fail_the_closed_form(name):
    old, new = MUTANTS[name]
    lib = _mutants.build_mutant(old, new)
    want = _closed_form(1)
    got = _mutants.moe_forward_with(lib, _layer(1), X)
    assert not np.allclose(got, want, rtol=1e-6, atol=1e-9), name
    # the unmutated source, built the same way, passes
    same = _mutants.build_mutant(old, old)
    np.testing.assert_allclose(_mutants.moe_forward_with(same, _layer(1), X), want, rtol=1e-14, atol=0.0)
