"""The fifth-generation tensor-core path (tcgen05 MMAs from 128-byte-swizzled
shared memory into tensor memory, tcgen05 loads back) on single tiles, against
the oracle's plain matrix product.  The batched expert kernels run their
contractions on this path.  Operands are small integers times powers of two,
so every product and every partial sum is exact in fp32 and the tensor core
must reproduce the oracle bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests._util import np_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("N", [16, 32, 48, 64, 128, 256])
def test_tcgen05_tile_matches_the_oracle(dfv, N, K):
    g = torch.Generator().manual_seed(N * 7 + K)
    a = (torch.randint(-8, 9, (128, K), generator=g).float() / 4).to(torch.bfloat16)
    b = (torch.randint(-8, 9, (N, K), generator=g).float() / 8).to(torch.bfloat16)
    d, st = dfv.selftest_tcgen05(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.matmul(oracle.BF16, np_of(a), np.ascontiguousarray(np_of(b).T)).astype(np.float32)
    got = d.cpu().numpy()
    assert np.array_equal(got, ref), float(np.max(np.abs(got - ref)))


def test_tcgen05_transposed_operand_would_be_caught(dfv):
    # a layout mistake that swaps rows for k would give A^T-like results: the
    # operands here make A . B^T differ from every such mix-up
    g = torch.Generator().manual_seed(3)
    a = (torch.randint(-8, 9, (128, 64), generator=g).float() / 4).to(torch.bfloat16)
    b = (torch.randint(-8, 9, (64, 64), generator=g).float() / 8).to(torch.bfloat16)
    d, st = dfv.selftest_tcgen05(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    ref = (a.double() @ b.double().T).float().numpy()
    assert np.array_equal(d.cpu().numpy(), ref)
    assert not np.array_equal(ref[:64, :64], (a.double()[:64] @ b.double()).float().numpy())
