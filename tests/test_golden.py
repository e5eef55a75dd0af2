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
                out.append([None if v == "-" else (float(int(v, 16)) if v.startswith("0x") else float(v))
                            for v in line.split()])
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


# ---------------------------------------------------------------- signed-zero multiply-add
# "Speculating on a Strix Halo (part 2)", section "Two bugs upstream".
SIGNED_ZERO = _rows("signed_zero_mma.txt")


def signed_zero_operands(neg_zero_row=None, fmt="f16"):
    """A and B of the page's 16x16 case as 16-bit patterns: column 12 of A is
    -1, row 12 of B is (j+1)/16, every other entry +0.0; with neg_zero_row set,
    that row of B holds -0.0 instead."""
    import torch
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    a = torch.zeros(16, 16, dtype=dt)
    a[:, 12] = -1.0
    b = torch.zeros(16, 16, dtype=dt)
    b[12, :] = torch.arange(1, 17, dtype=torch.float32) / 16
    if neg_zero_row is not None:
        assert neg_zero_row != 12
        b[neg_zero_row, :] = -0.0
    return a, b


def _bits(t):
    import torch
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("neg_zero_row", [None, 0, 7, 15])
def test_signed_zero_mma_exact_in_the_oracle(fmt, neg_zero_row):
    a, b = signed_zero_operands(neg_zero_row, fmt)
    if neg_zero_row is not None:  # the -0 run differs from the +0 run in 16 elements of B
        b0 = _bits(signed_zero_operands(None, fmt)[1])
        assert int((_bits(b) != b0).sum()) == 16
        assert np.all(_bits(a)[:, neg_zero_row] == 0)  # A is +0 in the column those entries meet
    code = oracle.F16 if fmt == "f16" else oracle.BF16
    d = oracle.matmul(code, _bits(a), _bits(b)).astype(np.float32)
    want = np.tile(-(np.arange(1, 17, dtype=np.float32)) / 16, (16, 1))
    assert np.array_equal(d.view(np.uint32), want.view(np.uint32))
    for i, j, value, bits in SIGNED_ZERO:
        assert d[int(i), int(j)] == value
        assert int(d[int(i), int(j):int(j) + 1].view(np.uint32)[0]) == int(bits)


@pytest.mark.parametrize("mistake", ["skips column 12", "transposes B"])
def test_signed_zero_case_catches_planted_matmul_mistakes(mistake):
    """Planted in a copy of the oracle's matrix product, each mistake misses
    the printed bits: skipping the one non-zero term leaves 0, a transposed B
    puts the column of (j+1)/16 values on the wrong axis."""
    from tests import _mutants
    loop = "for (int l = 0; l < L; ++l) acc += a[(size_t)i * L + l] * b[(size_t)l * N + j];"
    bad = {"skips column 12": "for (int l = 0; l < L; ++l) if (l != 12) acc += a[(size_t)i * L + l] * b[(size_t)l * N + j];",
           "transposes B": "for (int l = 0; l < L; ++l) acc += a[(size_t)i * L + l] * b[(size_t)j * N + l];"}[mistake]
    lib = _mutants.build_mutant(loop, bad)
    a, b = signed_zero_operands(None, "f16")
    d = _mutants.matmul_with(lib, oracle.F16, _bits(a), _bits(b)).astype(np.float32)
    assert any(d[int(i), int(j)] != value for i, j, value, _ in SIGNED_ZERO)


def test_signed_zero_fixture_bits_are_the_printed_values():
    for i, j, value, bits in SIGNED_ZERO:
        assert np.float32(value).view(np.uint32) == int(bits)
        assert value == -(j + 1) / 16
