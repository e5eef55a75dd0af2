"""Allocation-free acceptance entry point (collected last on purpose).

dfv_accept_greedy_noalloc serves callers that cannot allocate device memory:
its scratch is a fixed device array inside the library rather than a
caller-provided workspace.  It must compute exactly what dfv_accept_greedy
computes; this test calls both through the C ABI on the same inputs, twice in a
row with different inputs (the second call runs on the array as the first call
left it, so it shows that a call does not depend on what the array held)."""
from __future__ import annotations

import ctypes

import pytest
import torch

from speculative_decoding_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


def _call_both(dfv, logits, draft):
    lib = dfv.lib()
    rows, V = logits.shape
    k = rows - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = dfv.BF16 if logits.dtype == torch.bfloat16 else dfv.F32
    ws = dfv.alloc_workspace(dfv.accept_workspace_size(k, V))
    tau_a = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    com_a = torch.full((k + 1,), -7, dtype=torch.int32, device="cuda")
    tau_b = tau_a.clone()
    com_b = com_a.clone()
    st = lib.dfv_accept_greedy(ctypes.c_void_p(logits.data_ptr()), code, k, V, ctypes.c_void_p(draft.data_ptr()),
                               ctypes.c_void_p(tau_a.data_ptr()), ctypes.c_void_p(com_a.data_ptr()),
                               ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
    assert st == 0, lib.dfv_last_error_detail()
    st = lib.dfv_accept_greedy_noalloc(ctypes.c_void_p(logits.data_ptr()), code, k, V,
                                       ctypes.c_void_p(draft.data_ptr()), ctypes.c_void_p(tau_b.data_ptr()),
                                       ctypes.c_void_p(com_b.data_ptr()), stream)
    assert st == 0, lib.dfv_last_error_detail()
    torch.cuda.synchronize()
    return (tau_a, com_a), (tau_b, com_b)


def test_noalloc_acceptance_matches_workspace_entry_point_on_two_calls(dfv):
    cases = [(17, 151936, "bf16", 5), (5, 1024, "f32", 2)]
    for i, (rows, V, dt, n) in enumerate(cases):
        logits, toks = inputs.spiked_logits(rows, V, dt, 2.0, seed=70 + i, device="cuda")
        draft = toks[:rows - 1].clone()
        draft[n] = (draft[n] + 1) % V
        (ta, ca), (tb, cb) = _call_both(dfv, logits, draft)
        assert int(ta.item()) == n + 1
        assert torch.equal(ta, tb)
        assert torch.equal(ca, cb)
