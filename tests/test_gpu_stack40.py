"""The two full-size 40-layer stacks against the oracle, then greedy acceptance
on full-vocabulary logits: one verify cycle of the target ("Speculating on a
Strix Halo", sections "Speculative decoding" and "What the pieces cost"; part
2, "The verification cog": the verifier is the base model run over the draft).

* 40 Qwen3-A3B-like layers (d=2048, 128 experts, top-8, d_ff=768, bf16,
  independent seeded weights, 48 GB) and 40 mxfp4 layers (256 experts, top-8,
  d_ff=512, e2m1 + e8m0 per 32), pre-norm residual stack at k=16.
* Teacher forcing: every GPU layer is checked against the oracle fed the GPU's
  own input to that layer, so an error is caught in the layer that makes it.
  Rows whose normalised input has a near-tie in the router (gap between the
  K-th and (K+1)-th logit under 1e-3) are counted and left out of the output
  check: with a near-tie either expert set is a legitimate outcome of the
  summation order.
* The one-call stack over all 40 layers equals the layer-by-layer calls bit
  for bit in every launch mode (bf16: also as one persistent launch).
* Acceptance: logits[17, 151936] bf16 ~N(0, 2) with drafts planted from the
  oracle's argmax at Geometric(0.3) accepted lengths; tau and the committed
  tokens must equal the oracle's.

Each layer is copied to the host only for its own check, so the host never
holds more than one layer."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

N_LAYERS, K_BLOCK = 40, 16
TOL = {"bf16": 2e-2, "mxfp4": 5e-2}


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


def _threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _bf16_np(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("shape_name", ["bf16", "mxfp4"])
def test_stack40_teacher_forced_then_accept(dfv, shape_name):
    shape = inputs.A3B if shape_name == "bf16" else inputs.MXFP4
    tol = TOL[shape_name]
    seed0 = 4000 if shape_name == "bf16" else 5000
    lws = [inputs.make_layer(shape, seed=seed0 + l, device="cuda") for l in range(N_LAYERS)]
    Ls = [dfv.Layer(w) for w in lws]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, K_BLOCK) for L in Ls))
    x0 = inputs.make_hidden(K_BLOCK, shape.d, "bf16", seed=seed0 + 999, device="cuda")
    x = x0.clone()
    nthr = _threads()
    y = torch.empty(K_BLOCK, shape.d, dtype=torch.bfloat16, device="cuda")
    excluded, worst = 0, 0.0
    for l in range(N_LAYERS):
        xin = x.clone()
        dfv.moe_stack_forward([Ls[l]], x, ws)
        torch.cuda.synchronize()
        ol = oracle_layer(lws[l].to("cpu"))
        xin_np = np_of(xin)
        ref = oracle.stack_forward([ol], xin_np, nthreads=nthr)
        nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in oracle.rmsnorm(xin_np)], dtype=np.uint16)
        lg, _, _ = oracle.route(ol, nb)
        keep = topk_gap(lg, shape.top_k) >= 1e-3
        excluded += int((~keep).sum())
        if not keep.any():
            continue
        # the layer's MoE output on the normalised rows, against the oracle's
        dfv.moe_block_forward(Ls[l], torch.from_numpy(nb.view(np.int16)).view(torch.bfloat16).cuda(), ws, out=y)
        torch.cuda.synchronize()
        ref_moe = oracle.moe_forward(ol, nb, nthreads=nthr)[keep]
        rel = np.max(np.abs(y.double().cpu().numpy()[keep] - ref_moe)) / max(np.max(np.abs(ref_moe)), 1e-30)
        worst = max(worst, rel)
        assert rel <= tol, "layer %d: MoE output error %.3g of max|ref|" % (l, rel)
        # the residual update: x_out = bf16(x_in + MoE(bf16(RMSNorm(x_in)))); each
        # element may differ from the oracle's by the MoE tolerance plus one bf16
        # spacing at its own magnitude (the two sums can round to neighbours)
        got = x.double().cpu().numpy()[keep]
        refd = _bf16_np(ref)[keep]
        delta_ref = refd - xin.double().cpu().numpy()[keep]
        scale = max(np.max(np.abs(delta_ref)), 1e-30)
        mag = np.maximum(np.abs(refd), 2.0 ** -126)
        ulp = np.exp2(np.floor(np.log2(mag)) - 7)
        bad = np.abs(got - refd) > tol * scale + ulp
        assert not bad.any(), "layer %d: %d residual elements off" % (l, int(bad.sum()))
        del ol
    print("\n%s stack40: %d of %d rows excluded as near-ties; worst layer MoE error %.2e of max|ref|"
          % (shape_name, excluded, N_LAYERS * K_BLOCK, worst))
    assert excluded <= N_LAYERS * K_BLOCK // 4
    assert dfv.read_device_error(ws) == 0

    # the one-call stack equals the layer-by-layer calls, in every launch mode
    # (bf16 layers: mode 2 is one persistent launch for all 40 layers)
    xs = x0.clone()
    dfv.moe_stack_forward(Ls, xs, ws)
    torch.cuda.synchronize()
    assert torch.equal(xs, x)
    for mode, want in ((2, 3 if shape_name == "bf16" else 1), (0, 1)):
        dfv.set_stack_launch(mode)
        try:
            xp = x0.clone()
            dfv.moe_stack_forward(Ls, xp, ws)
            torch.cuda.synchronize()
            path = dfv.last_layer_path()
        finally:
            dfv.set_stack_launch(1)
        assert path == want
        assert torch.equal(xp, x)
    del Ls, lws

    # acceptance on the full vocabulary after the stack
    V = 151936
    aws = dfv.alloc_workspace(dfv.accept_workspace_size(K_BLOCK, V))
    ns = inputs.geometric_accept_lengths(4, 0.3, K_BLOCK - 1, seed=seed0 + 7)
    for i, n in enumerate(ns.tolist()):
        lg = inputs.make_logits(K_BLOCK + 1, V, "bf16", 2.0, seed=seed0 + 100 + i)
        a = oracle.argmax_rows(np_of(lg))
        draft = inputs.plant_draft(torch.from_numpy(a), int(n), V, seed=seed0 + 200 + i)
        tau, com = dfv.accept_greedy(lg.cuda(), draft.cuda(), aws)
        torch.cuda.synchronize()
        tau_o, com_o = oracle.accept_greedy(np_of(lg), draft.numpy())
        assert int(tau.item()) == tau_o == int(n) + 1
        assert np.array_equal(com.cpu().numpy(), com_o)
