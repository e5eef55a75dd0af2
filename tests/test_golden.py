"""Values the pages print, kept as fixtures under tests/golden/ with their
citations, checked against the oracle's acceptance and the bench's arithmetic.
CPU only."""
from __future__ import annotations

import math
import os
import sys

import numpy as np
import pytest

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import np_of

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _rows(name):
    out = []
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([None if v == "-" else float(v) for v in line.split()])
    return out


GEOM = _rows("geometric_acceptance.txt")


@pytest.mark.parametrize("p,depth,tau,tol,none,one", GEOM)
def test_geometric_acceptance_closed_form(p, depth, tau, tol, none, one):
    # tau = 1 + E[accepted prefix] = sum_{i=0}^{depth} p^i
    closed = (1 - p ** (int(depth) + 1)) / (1 - p)
    assert abs(closed - tau) <= tol
    if none is not None:
        assert abs((1 - p) - none) < 1e-9 and abs(p * (1 - p) - one) < 1e-9


@pytest.mark.parametrize("p,depth,tau,tol,none,one", [r for r in GEOM if r[0] == 0.80 and r[1] == 15])
def test_geometric_acceptance_through_the_oracle(p, depth, tau, tol, none, one):
    """Cycles whose drafts match the target's greedy tokens for a geometric
    number of positions: the oracle's committed lengths reproduce the printed
    mean and shares within sampling error."""
    k, V, n_cycles = int(depth), 97, 4000
    lg, tokens = inputs.spiked_logits(k + 1, V, "f32", 1.0, seed=41)
    lg_np = np_of(lg)
    assert np.array_equal(oracle.argmax_rows(lg_np), tokens.numpy())
    accepted = inputs.geometric_accept_lengths(n_cycles, 1 - p, k, seed=42).tolist()
    taus = []
    for c, n in enumerate(accepted):
        draft = inputs.plant_draft(tokens, int(n), V, seed=1000 + c)
        t, _ = oracle.accept_greedy(lg_np, draft.numpy())
        taus.append(t)
    taus = np.array(taus, dtype=np.float64)
    sem = taus.std() / math.sqrt(n_cycles)
    assert abs(taus.mean() - tau) <= tol + 4 * sem
    assert abs((taus == 1).mean() - none) <= 4 * math.sqrt(none * (1 - none) / n_cycles)
    assert abs((taus == 2).mean() - one) <= 4 * math.sqrt(one * (1 - one) / n_cycles)


@pytest.mark.parametrize("gb,ms,gbs", _rows("effective_bandwidth.txt"))
def test_effective_bandwidth_arithmetic(gb, ms, gbs):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.achieved_gbs(gb * 1e9, ms) == pytest.approx(gbs, rel=0.02)
