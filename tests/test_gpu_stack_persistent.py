"""The persistent stack launch: all layers of a pre-norm residual stack in one
cooperative launch ("Speculating on a Strix Halo (part 2)", section "The
verification cog": each layer of the target pays its own fixed cost, and the
decode of one token pays it in full).

The stack kernel runs the same per-layer phases as the one-launch-per-layer
path, so the two must agree bit for bit; the per-layer path is itself checked
against the oracle layer by layer (tests/test_gpu_parity.py), and so is the
stack kernel here, one layer per launch.  Covered here: block sizes on
both sides of the 8-token split, a shared expert, every gate/up staging mode,
stacks longer than one launch holds (48 layers), repeated calls on one
workspace (the grid-barrier count must be reset by every launch), the default
launch mode's choice by block size, and the fallback for stacks whose layers
differ in shape."""
from __future__ import annotations

import pytest
import torch

import numpy as np

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

SMALL = inputs.LayerShape(d=512, n_experts=32, top_k=4, d_ff=128)
SMALL_SHARED = inputs.LayerShape(d=512, n_experts=32, top_k=4, d_ff=128, n_shared=1)
TINY_BF16 = inputs.LayerShape(d=256, n_experts=16, top_k=2, d_ff=64)


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


def _layers(dfv, shape, n, seed):
    lws = [inputs.make_layer(shape, seed=seed + l, device="cuda") for l in range(n)]
    return lws, [dfv.Layer(w) for w in lws]


def _run(dfv, Ls, x0, ws, persistent):
    """persistent: True = one launch for the stack at any k (mode 2), False = one launch per layer."""
    dfv.set_stack_launch(2 if persistent else 0)
    try:
        x = x0.clone()
        dfv.moe_stack_forward(Ls, x, ws)
        torch.cuda.synchronize()
        path = dfv.last_layer_path()
    finally:
        dfv.set_stack_launch(1)
    return x, path


@pytest.mark.parametrize("shape_name", ["small", "shared"])
@pytest.mark.parametrize("k", [1, 3, 8, 9, 16])
def test_persistent_equals_per_layer_launches(dfv, shape_name, k):
    shape = SMALL if shape_name == "small" else SMALL_SHARED
    lws, Ls = _layers(dfv, shape, 7, seed=7000 + k)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x0 = inputs.make_hidden(k, shape.d, "bf16", seed=7100 + k, device="cuda")
    ref, p0 = _run(dfv, Ls, x0, ws, False)
    got, p1 = _run(dfv, Ls, x0, ws, True)
    assert p0 == 1 and p1 == 3
    assert torch.equal(got, ref)
    assert not torch.equal(got, x0)
    assert dfv.read_device_error(ws) == 0


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_persistent_every_staging_mode(dfv, mode):
    lws, Ls = _layers(dfv, SMALL, 5, seed=7200)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x0 = inputs.make_hidden(16, SMALL.d, "bf16", seed=7201, device="cuda")
    ref, _ = _run(dfv, Ls, x0, ws, False)
    dfv.set_staging(mode)
    try:
        got, path = _run(dfv, Ls, x0, ws, True)
        used = dfv.last_staging()
    finally:
        dfv.set_staging(3)
    assert path == 3 and used <= mode
    assert torch.equal(got, ref)


def test_persistent_longer_than_one_launch(dfv):
    """50 layers: one launch of 48 layers, then one of 2."""
    lws, Ls = _layers(dfv, TINY_BF16, 50, seed=7300)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    for k in (1, 16):
        x0 = inputs.make_hidden(k, TINY_BF16.d, "bf16", seed=7301 + k, device="cuda")
        ref, _ = _run(dfv, Ls, x0, ws, False)
        got, path = _run(dfv, Ls, x0, ws, True)
        assert path == 3
        assert torch.equal(got, ref)
    assert dfv.read_device_error(ws) == 0


def test_persistent_repeated_calls_one_workspace(dfv):
    lws, Ls = _layers(dfv, SMALL, 4, seed=7400)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x0 = inputs.make_hidden(16, SMALL.d, "bf16", seed=7401, device="cuda")
    first, _ = _run(dfv, Ls, x0, ws, True)
    for _ in range(5):
        again, path = _run(dfv, Ls, x0, ws, True)
        assert path == 3
        assert torch.equal(again, first)
    # chained without a host sync in between
    xs = [x0.clone() for _ in range(4)]
    dfv.set_stack_launch(2)
    try:
        for x in xs:
            dfv.moe_stack_forward(Ls, x, ws)
        torch.cuda.synchronize()
    finally:
        dfv.set_stack_launch(1)
    for x in xs:
        assert torch.equal(x, first)
    assert dfv.read_device_error(ws) == 0


def test_default_mode_persistent_up_to_8_tokens(dfv):
    """The default launch mode takes the persistent kernel for eager calls with
    k <= 8 and one launch per layer above; every mode gives the same bits."""
    lws, Ls = _layers(dfv, SMALL, 3, seed=7450)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    for k, want in ((1, 3), (8, 3), (9, 1), (16, 1)):
        x0 = inputs.make_hidden(k, SMALL.d, "bf16", seed=7451 + k, device="cuda")
        x = x0.clone()
        dfv.moe_stack_forward(Ls, x, ws)
        torch.cuda.synchronize()
        assert dfv.last_layer_path() == want
        ref, _ = _run(dfv, Ls, x0, ws, False)
        assert torch.equal(x, ref)


def test_mixed_shapes_fall_back_to_per_layer_launches(dfv):
    a, La = _layers(dfv, SMALL, 2, seed=7500)
    b, Lb = _layers(dfv, inputs.LayerShape(d=512, n_experts=48, top_k=4, d_ff=128), 2, seed=7510)
    Ls = [La[0], Lb[0], La[1], Lb[1]]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16) for L in Ls))
    x0 = inputs.make_hidden(16, 512, "bf16", seed=7501, device="cuda")
    ref, p0 = _run(dfv, Ls, x0, ws, False)
    got, p1 = _run(dfv, Ls, x0, ws, True)
    assert p0 == 1 and p1 == 1
    assert torch.equal(got, ref)


def test_a3b_stack_persistent_equals_per_layer(dfv):
    """Four full-size Qwen3-A3B-like layers at k = 1 and k = 16."""
    lws, Ls = _layers(dfv, inputs.A3B, 4, seed=7600)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    for k in (1, 16):
        x0 = inputs.make_hidden(k, inputs.A3B.d, "bf16", seed=7601 + k, device="cuda")
        ref, _ = _run(dfv, Ls, x0, ws, False)
        got, path = _run(dfv, Ls, x0, ws, True)
        assert path == 3
        assert torch.equal(got, ref)
    assert dfv.read_device_error(ws) == 0


@pytest.mark.parametrize("k", [4, 16])
def test_stack_kernel_teacher_forced_against_oracle(dfv, k):
    """Each layer through the stack kernel (a one-layer persistent launch), on
    the GPU's own input to that layer, against the oracle's pre-norm residual
    layer: x_out = bf16(x + MoE(bf16(RMSNorm(x)))).  Rows with a near-tie in
    the router (gap under 1e-3) are left out of the comparison."""
    shape = SMALL_SHARED if k == 4 else SMALL
    n_layers = 4
    lws, Ls = _layers(dfv, shape, n_layers, seed=7700 + k)
    ols = [oracle_layer(w.to("cpu")) for w in lws]
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x = inputs.make_hidden(k, shape.d, "bf16", seed=7701 + k, device="cuda")
    excluded = 0
    dfv.set_stack_launch(2)
    try:
        for l in range(n_layers):
            xin = x.clone()
            dfv.moe_stack_forward([Ls[l]], x, ws)
            torch.cuda.synchronize()
            assert dfv.last_layer_path() == 3
            xin_np = np_of(xin)
            ref = oracle.stack_forward([ols[l]], xin_np)
            nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in oracle.rmsnorm(xin_np)], dtype=np.uint16)
            lg, _, _ = oracle.route(ols[l], nb)
            keep = topk_gap(lg, shape.top_k) >= 1e-3
            excluded += int((~keep).sum())
            got = x.double().cpu().numpy()[keep]
            refd = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy()[keep]
            delta_ref = refd - xin.double().cpu().numpy()[keep]
            # the MoE tolerance on the update, plus one bf16 spacing at each
            # element's own magnitude (x + update rounds once to bf16 on each
            # side, and two close sums can round to neighbours)
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(refd), 2.0 ** -126))) - 7)
            bad = np.abs(got - refd) > 2e-2 * max(np.max(np.abs(delta_ref)), 1e-30) + ulp
            assert not bad.any(), "layer %d: %d elements off" % (l, int(bad.sum()))
    finally:
        dfv.set_stack_launch(1)
    assert excluded <= n_layers * k // 4
    assert dfv.read_device_error(ws) == 0


def test_default_mode_launches_per_layer_inside_a_graph(dfv):
    """Captured in a CUDA graph, the default mode launches per layer even at
    k = 1 (chained launches are the faster choice there); the replay equals
    the eager persistent call."""
    lws, Ls = _layers(dfv, SMALL, 3, seed=7480)
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x0 = inputs.make_hidden(1, SMALL.d, "bf16", seed=7481, device="cuda")
    ref = x0.clone()
    dfv.moe_stack_forward(Ls, ref, ws)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == 3
    x = x0.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dfv.moe_stack_forward(Ls, x, ws, stream=s)
    assert dfv.last_layer_path() == 1
    x.copy_(x0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x, ref)
