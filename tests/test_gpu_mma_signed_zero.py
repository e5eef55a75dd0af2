"""The tensor-core fragment path of the expert kernels on the 16x16 case of
"Speculating on a Strix Halo (part 2)", section "Two bugs upstream": column 12
of A is -1, row 12 of B is (j+1)/16, everything else zero, so D[i][j] is
exactly -(j+1)/16.  The page prints the first values' binary32 patterns
(tests/golden/signed_zero_mma.txt).  Both the +0 run and runs with one row of
B's zeros stored as -0.0 must return those bits, through the bf16 kernels'
MMA helper and through the mxfp4 kernels' fp16 one, and agree bit for bit with
the oracle's plain matrix product."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests.test_golden import SIGNED_ZERO, _bits, signed_zero_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("neg_zero_row", [None, 0, 3, 8, 11, 13, 15])
def test_signed_zero_case_is_exact_through_the_mma_path(dfv, fmt, neg_zero_row):
    a, b = signed_zero_operands(neg_zero_row, fmt)
    d = dfv.selftest_mma(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    got = d.cpu().numpy()
    want = np.tile(-(np.arange(1, 17, dtype=np.float32)) / 16, (16, 1))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for i, j, value, bits in SIGNED_ZERO:
        assert int(got[int(i), int(j):int(j) + 1].view(np.uint32)[0]) == int(bits)
    code = oracle.F16 if fmt == "f16" else oracle.BF16
    ref = oracle.matmul(code, _bits(a), _bits(b)).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_mma_path_matches_the_oracle_on_random_operands(dfv, fmt):
    # small integers times powers of two: every product and partial sum is
    # exact in fp32, so the tensor core must reproduce the oracle exactly
    g = torch.Generator().manual_seed(5)
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    a = (torch.randint(-8, 9, (16, 16), generator=g).float() / 4).to(dt)
    b = (torch.randint(-8, 9, (16, 16), generator=g).float() / 8).to(dt)
    d = dfv.selftest_mma(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    code = oracle.F16 if fmt == "f16" else oracle.BF16
    ref = oracle.matmul(code, _bits(a), _bits(b)).astype(np.float32)
    assert np.array_equal(d.cpu().numpy(), ref)
    assert not np.array_equal(ref, ref.T)  # a transposed operand would be caught
