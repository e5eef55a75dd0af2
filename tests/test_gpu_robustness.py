"""Failure detection and stale-data checks on the GPU, with no fault.

* Stale workspace contents: every data section of the workspace (logits,
  routing tables, h, ys, staging) is filled with NaN, negative-zero or random
  bytes before a call; the outputs must equal those of a zero-filled workspace
  bit for bit.  Only the 8 KB of counters at the start must be zero (the ABI's
  rule).  (Part 2 of "Speculating on a Strix Halo" traces a verification bug
  to stale values read from a buffer; this is the same check on ours.)
* Guard bands: the rows just before and after an output block stay untouched.
* Bounded waits: the self-test entry point makes an mbarrier wait and a grid
  barrier wait run out; each must set its error bit and return, and the
  context must still compute a correct layer afterwards."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import hidden_without_near_ties, np_of, oracle_layer

pytestmark = pytest.mark.gpu

COUNTER_BYTES = 8192  # the counters at fixed offsets, first in every workspace


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


def _fill(ws: torch.Tensor, kind: str, seed: int):
    """ws is a uint8 tensor: keep the counters zero, overwrite the rest."""
    body = ws[COUNTER_BYTES:]
    if kind == "nan":
        body.fill_(0xFF)  # fp32 / bf16 NaN, int32 -1
    elif kind == "negzero":
        body.view(torch.int32)[:] = torch.tensor(-2 ** 31, dtype=torch.int32)  # fp32 -0.0
    else:
        g = torch.Generator(device=ws.device)
        g.manual_seed(seed)
        body.copy_(torch.randint(0, 256, body.shape, generator=g, device=ws.device, dtype=torch.int32).to(torch.uint8))
    ws[:COUNTER_BYTES].zero_()


LAYERS = [
    ("bf16", inputs.LayerShape(d=512, n_experts=40, top_k=8, d_ff=160)),
    ("bf16-shared", inputs.LayerShape(d=512, n_experts=40, top_k=8, d_ff=160, n_shared=1)),
    ("mxfp4", inputs.LayerShape(d=1024, n_experts=16, top_k=4, d_ff=192, w_dtype="mxfp4")),
]


@pytest.mark.parametrize("name,shape", LAYERS, ids=[n for n, _ in LAYERS])
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "multi"])
@pytest.mark.parametrize("k", [1, 16])
def test_stale_workspace_contents_do_not_change_outputs(dfv, name, shape, fused, k):
    lw = inputs.make_layer(shape, seed=31, device="cuda")
    L = dfv.Layer(lw)
    x = inputs.make_hidden(k, shape.d, "bf16", seed=32, device="cuda")
    nbytes = dfv.workspace_size(L, 16)
    dfv.set_path(fused)
    try:
        ws = dfv.alloc_workspace(nbytes)
        idx0 = torch.empty(k, shape.top_k, dtype=torch.int32, device="cuda")
        ref = dfv.moe_block_forward(L, x, ws, topk_idx=idx0).clone()
        torch.cuda.synchronize()
        assert dfv.read_device_error(ws) == 0
        for i, kind in enumerate(("nan", "negzero", "random")):
            _fill(ws, kind, seed=33 + i)
            idx = torch.empty_like(idx0)
            out = dfv.moe_block_forward(L, x, ws, topk_idx=idx)
            torch.cuda.synchronize()
            assert dfv.read_device_error(ws) == 0, kind
            assert torch.equal(idx, idx0), kind
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), kind
    finally:
        dfv.set_path(True)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "multi"])
def test_output_guard_bands_untouched(dfv, fused):
    shape = inputs.LayerShape(d=512, n_experts=40, top_k=8, d_ff=160, n_shared=1)
    lw = inputs.make_layer(shape, seed=34, device="cuda")
    L = dfv.Layer(lw)
    k = 9
    x = inputs.make_hidden(k, 512, "bf16", seed=35, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    canary = torch.full((k + 2, 512), 12345, dtype=torch.int16, device="cuda")  # bf16 bits 0x3039
    out = canary.view(torch.bfloat16)[1:k + 1]
    dfv.set_path(fused)
    try:
        dfv.moe_block_forward(L, x, ws, out=out)
        torch.cuda.synchronize()
    finally:
        dfv.set_path(True)
    assert torch.all(canary[0] == 12345) and torch.all(canary[k + 1] == 12345)
    ref = oracle.moe_forward(oracle_layer(lw.to("cpu")), np_of(x))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 2e-2 * np.max(np.abs(ref))


def test_bounded_waits_give_up_report_and_leave_the_context_usable(dfv):
    shape = inputs.LayerShape(d=512, n_experts=32, top_k=4, d_ff=128)
    lw = inputs.make_layer(shape, seed=36, device="cuda")
    L = dfv.Layer(lw)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    t0 = time.perf_counter()
    dfv.selftest_bounded_waits(ws)
    err = dfv.read_device_error(ws)
    dt = time.perf_counter() - t0
    assert err & dfv.DEVERR_STAGE_WAIT, hex(err)
    assert err & dfv.DEVERR_GRID_WAIT, hex(err)
    assert 3.5 < dt < 60.0  # two waits of about 2 s each
    # the same context, a zero-filled workspace: a correct layer
    ws.zero_()
    ol = oracle_layer(lw.to("cpu"))
    x = hidden_without_near_ties(ol, 16, "bf16", seed=37)
    out = dfv.moe_block_forward(L, x.cuda(), ws)
    torch.cuda.synchronize()
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 2e-2 * np.max(np.abs(ref))
