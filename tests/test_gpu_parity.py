"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing decisions (top-K indices, woken set, offsets, gather order) and tau
must be bit-exact; expert outputs within max|err| <= 2e-2 * max|ref| for bf16
and fp32 weights (fp32 accumulation on both sides).  Inputs are seeded and
drawn without near-ties (gap between the K-th and (K+1)-th router logit at
least 1e-3), so the routing decision is robust to summation order."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import hidden_without_near_ties, np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


def _max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(got.astype(np.float64) - ref)) / max(scale, 1e-30))


def _gpu_out_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _check_routing(dfv, L, ol, x, ws):
    r = dfv.route_topk(L, x, ws)
    torch.cuda.synchronize()
    _, idx, w = oracle.route(ol, np_of(x))
    wk, offs, gat = oracle.woken(idx, ol.n_experts)
    W = int(r["n_woken"].item())
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert W == len(wk)
    assert np.array_equal(r["woken"].cpu().numpy()[:W], wk)
    assert np.array_equal(r["offsets"].cpu().numpy()[:W + 1], offs)
    assert np.array_equal(r["gather"].cpu().numpy(), gat)
    assert np.allclose(r["topk_w"].cpu().numpy(), w, rtol=1e-5, atol=1e-6)
    return W


SMALL = [
    # d, E, K, I : several tiles, ragged warp splits and a ragged down tile (d % 64 != 0)
    (352, 24, 3, 96),
    (512, 40, 8, 160),
    (256, 8, 8, 64),  # K == E: every row wakes every expert
    (96, 8, 1, 64),   # top-1 routing, fewer experts than a warp has lanes
    (64, 4, 2, 32),   # narrow rows: fewer 32-column chunks than consumer warps
]


@pytest.fixture(params=["fused", "multi"])
def path(request, dfv):
    dfv.set_path(request.param == "fused")
    yield request.param
    dfv.set_path(True)


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("k", [1, 3, 8, 9, 16])
def test_bf16_layer_parity_small(dfv, path, shape, k):
    d, E, K, I = shape
    s = inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I)
    lw = inputs.make_layer(s, seed=100 + k)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=200 + k)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    _check_routing(dfv, L, ol, xg, ws)
    out = dfv.moe_block_forward(L, xg, ws)
    torch.cuda.synchronize()
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=8)
    assert _max_rel_err(_gpu_out_np(out), ref) <= TOL_BF16


WIDE = [
    # d, E, K, I: rows wider than 1024 (2-4 gate/up stages per unit, row copies
    # when d is not a multiple of 256); a repeated-token block gives experts up
    # to 16 tokens, so the staged x rows 8..15 are in use
    (1056, 16, 4, 64),
    (2304, 16, 4, 128),
    (2560, 12, 2, 192),
]


@pytest.mark.parametrize("shape", WIDE)
@pytest.mark.parametrize("k,mode", [(16, "repeated"), (12, "independent"), (1, "independent")])
def test_bf16_wide_rows(dfv, path, shape, k, mode):
    d, E, K, I = shape
    lw = inputs.make_layer(inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I), seed=d + 7 * k, device="cuda")
    ol = oracle_layer(lw.to("cpu"))
    L = dfv.Layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=d + k, mode=mode)
    xg = x.cuda()
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    _check_routing(dfv, L, ol, xg, ws)
    out = dfv.moe_block_forward(L, xg, ws)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == (1 if path == "fused" else 0), dfv.fused_unavailable_reason()
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    assert _max_rel_err(_gpu_out_np(out), ref) <= TOL_BF16
    if k > 1 and path == "fused":
        # the block's rows equal single-token calls bit for bit
        for t in (0, k - 1):
            row = dfv.moe_block_forward(L, xg[t:t + 1].contiguous(), ws)
            torch.cuda.synchronize()
            assert torch.equal(row[0], out[t])


WIDE_FF = [
    # d, E, K, I: expert intermediates wider than the single-launch kernel
    # takes (d_ff > 768), on the general path: ragged unit counts, top-2/4
    (512, 16, 4, 1024),
    (2048, 12, 4, 1408),
    (4096, 8, 2, 1536),
]


@pytest.mark.parametrize("shape", WIDE_FF)
@pytest.mark.parametrize("k,mode", [(16, "repeated"), (9, "independent"), (1, "independent")])
def test_bf16_wide_intermediate_general_path(dfv, shape, k, mode):
    d, E, K, I = shape
    lw = inputs.make_layer(inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I), seed=I + 7 * k, device="cuda")
    ol = oracle_layer(lw.to("cpu"))
    L = dfv.Layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=I + k, mode=mode)
    xg = x.cuda()
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    _check_routing(dfv, L, ol, xg, ws)
    out = dfv.moe_block_forward(L, xg, ws)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == 0  # the single-launch kernel does not take d_ff > 768
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    assert _max_rel_err(_gpu_out_np(out), ref) <= TOL_BF16
    if k > 1:
        for t in (0, k - 1):
            row = dfv.moe_block_forward(L, xg[t:t + 1].contiguous(), ws)
            torch.cuda.synchronize()
            assert torch.equal(row[0], out[t])


@pytest.mark.parametrize("k", [1, 4])
def test_tiny_fp32_config(dfv, k):
    lw = inputs.make_layer(inputs.TINY, seed=1)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "f32", seed=2)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    _check_routing(dfv, L, ol, xg, ws)
    out = dfv.moe_block_forward(L, xg, ws)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(ol, np_of(x))
    assert _max_rel_err(_gpu_out_np(out), ref) <= TOL_BF16


@pytest.fixture(scope="module")
def a3b(dfv):
    lw = inputs.make_layer(inputs.A3B, seed=7, device="cuda")
    return lw, oracle_layer(lw.to("cpu")), dfv.Layer(lw)


@pytest.mark.parametrize("k,mode", [(1, "independent"), (16, "independent"), (16, "repeated"), (7, "independent")])
def test_a3b_layer_full_size(dfv, a3b, path, k, mode):
    lw, ol, L = a3b
    x = hidden_without_near_ties(ol, k, "bf16", seed=300 + k, mode=mode)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    W = _check_routing(dfv, L, ol, xg, ws)
    assert W <= min(128, 8 * k)
    if k == 1:
        assert W == 8
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, xg, ws, n_woken=nw)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == (1 if path == "fused" else 0), dfv.fused_unavailable_reason()
    assert int(nw.item()) == W
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    assert _max_rel_err(_gpu_out_np(out), ref) <= TOL_BF16


def test_block_rows_equal_single_token_calls(dfv, a3b, path):
    """Losslessness on the GPU: row t of a 16-row block is bit-identical to the
    k=1 call on that row (fixed per-element summation order)."""
    lw, ol, L = a3b
    x = inputs.make_hidden(16, 2048, "bf16", seed=11, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    blk = dfv.moe_block_forward(L, x, ws).clone()
    for t in range(16):
        row = dfv.moe_block_forward(L, x[t:t + 1].contiguous(), ws)
        assert torch.equal(row[0], blk[t]), "row %d differs" % t


@pytest.mark.parametrize("norm_topk", [1, 0])
def test_route_topk_rows_equal_single_row_calls(dfv, norm_topk):
    """The routing launch has 512 threads for k > 8 (a warp per row in its top-K
    tail) and 256 for k <= 8; a row's experts and weights must not depend on
    which one ran it, nor on the other rows of the block."""
    s = dataclasses.replace(inputs.A3B, n_experts=256, d_ff=64, norm_topk=norm_topk)  # routing only
    lw = inputs.make_layer(s, seed=21, device="cuda")
    L = dfv.Layer(lw)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    x = inputs.make_hidden(16, s.d, "bf16", seed=22, device="cuda")
    blk = dfv.route_topk(L, x, ws)
    idx, w = blk["topk_idx"].clone(), blk["topk_w"].clone()
    for k in (1, 8, 9):
        part = dfv.route_topk(L, x[:k].contiguous(), ws)
        assert torch.equal(part["topk_idx"], idx[:k]), k
        assert torch.equal(part["topk_w"], w[:k]), k
    assert dfv.read_device_error(ws) == 0


def test_identical_rows_wake_one_set(dfv, a3b):
    lw, ol, L = a3b
    x = inputs.make_hidden(1, 2048, "bf16", seed=12, device="cuda").repeat(16, 1).contiguous()
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    r = dfv.route_topk(L, x, ws)
    assert int(r["n_woken"].item()) == 8
    out = dfv.moe_block_forward(L, x, ws)
    assert all(torch.equal(out[0], out[t]) for t in range(16))


def test_signed_zeros_do_not_change_results(dfv):
    """Zero-valued inputs of either sign give bit-identical outputs (masked or
    zero lanes must not leak into the result through the sign of zero)."""
    s = inputs.LayerShape(d=256, n_experts=16, top_k=4, d_ff=64)
    lw = inputs.make_layer(s, seed=13, device="cuda")
    x = inputs.make_hidden(5, 256, "bf16", seed=13, device="cuda")
    x[:, ::3] = 0.0
    xn = x.clone()
    xn[:, ::3] = -0.0
    wg2 = lw.w_gate.clone()
    wg2[:, :, ::5] = 0.0
    wg3 = wg2.clone()
    wg3[:, :, ::5] = -0.0
    outs = []
    for xx, wg in ((x, wg2), (xn, wg3)):
        L = dfv.Layer(inputs.LayerWeights(s, lw.w_router, wg, lw.w_up, lw.w_down))
        ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
        outs.append(dfv.moe_block_forward(L, xx, ws).clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_workspace_reuse_and_host_variant(dfv, a3b, path):
    lw, ol, L = a3b
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xa = inputs.make_hidden(16, 2048, "bf16", seed=14, device="cuda")
    xb = inputs.make_hidden(3, 2048, "bf16", seed=15, device="cuda")
    a1 = dfv.moe_block_forward(L, xa, ws).clone()
    dfv.moe_block_forward(L, xb, ws)
    a2 = dfv.moe_block_forward(L, xa, ws).clone()
    assert torch.equal(a1, a2)
    hx = xa.cpu().pin_memory()
    ho = torch.empty_like(hx).pin_memory()
    dfv.moe_block_forward_host(L, hx, ho, ws)
    torch.cuda.synchronize()
    assert torch.equal(ho, a1.cpu())


# ---------------------------------------------------------------- acceptance


def _accept_case(dfv, logits_cpu, n_plant, seed):
    a = oracle.argmax_rows(np_of(logits_cpu))
    V = logits_cpu.shape[1]
    draft = inputs.plant_draft(torch.from_numpy(a), n_plant, V, seed)
    tau_o, com_o = oracle.accept_greedy(np_of(logits_cpu), draft.numpy())
    ws = dfv.alloc_workspace(dfv.accept_workspace_size(16, V))
    tau, com = dfv.accept_greedy(logits_cpu.cuda(), draft.cuda(), ws)
    torch.cuda.synchronize()
    assert int(tau.item()) == tau_o == n_plant + 1
    assert np.array_equal(com.cpu().numpy(), com_o)


@pytest.mark.parametrize("n", [0, 1, 3, 4])
def test_accept_tiny_fp32(dfv, n):
    lg = inputs.make_logits(5, 1024, "f32", 1.0, seed=20 + n)
    _accept_case(dfv, lg, n, seed=n)


@pytest.mark.parametrize("n", [0, 2, 7, 15, 16])
def test_accept_bf16_full_vocab(dfv, n):
    lg = inputs.make_logits(17, 151936, "bf16", 2.0, seed=30 + n)
    _accept_case(dfv, lg, n, seed=n)


def test_accept_ties_and_ragged_vocab(dfv):
    for V in (2, 7, 1000, 4099):
        lg = inputs.make_logits(4, V, "bf16", 2.0, seed=V)
        lg[1, :] = 0.0
        lg[1, V // 2:] = -0.0
        if V > 3:
            lg[2, [1, V - 1]] = 50.0
        _accept_case(dfv, lg, 1, seed=V)


def test_accept_geometric_planted_lengths(dfv):
    ns = inputs.geometric_accept_lengths(12, 0.3, 15, seed=40)
    for i, n in enumerate(ns.tolist()):
        lg = inputs.make_logits(17, 151936, "bf16", 2.0, seed=400 + i)
        _accept_case(dfv, lg, n, seed=i)


# ---------------------------------------------------------------- stack


def test_stack_teacher_forced_and_fused(dfv, path):
    """Pre-norm residual stack: each GPU layer checked against the oracle on the
    GPU's own layer input; the one-call stack equals the layer-by-layer calls."""
    shape = inputs.LayerShape(d=512, n_experts=32, top_k=4, d_ff=128)
    n_layers, k = 6, 16
    lws = [inputs.make_layer(shape, seed=500 + l, device="cuda") for l in range(n_layers)]
    Ls = [dfv.Layer(w) for w in lws]
    ols = [oracle_layer(w.to("cpu")) for w in lws]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16) for L in Ls))
    x0 = inputs.make_hidden(k, 512, "bf16", seed=501, device="cuda")
    x = x0.clone()
    excluded = 0
    for l in range(n_layers):
        xin = x.clone()
        dfv.moe_stack_forward([Ls[l]], x, ws)
        torch.cuda.synchronize()
        xin_np = np_of(xin)
        ref = oracle.stack_forward([ols[l]], xin_np)
        # rows whose normalised input has a near-tie in the router are only
        # compared where the routing agrees (a flip there is a legitimate
        # rounding-order outcome, not an error)
        nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in oracle.rmsnorm(xin_np)], dtype=np.uint16)
        lg, _, _ = oracle.route(ols[l], nb)
        keep = topk_gap(lg, shape.top_k) >= 1e-3
        excluded += int((~keep).sum())
        got = _gpu_out_np(x)[keep]
        refd = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy()[keep]
        delta_ref = refd - _gpu_out_np(xin)[keep]
        bound = TOL_BF16 * max(np.max(np.abs(delta_ref)), 1e-30) + np.max(np.abs(refd)) * 2 ** -8
        assert np.max(np.abs(got - refd)) <= bound, "layer %d" % l
    assert excluded <= n_layers * k // 4
    xs = x0.clone()
    dfv.moe_stack_forward(Ls, xs, ws)
    torch.cuda.synchronize()
    assert torch.equal(xs, x)


def test_fused_and_multikernel_paths_agree(dfv, a3b):
    """Both kernel paths compute the same function: equal routing, outputs
    within the bf16 tolerance of each other."""
    lw, ol, L = a3b
    x = inputs.make_hidden(16, 2048, "bf16", seed=16, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    outs, idxs = [], []
    for fused in (True, False):
        dfv.set_path(fused)
        idx = torch.empty(16, 8, dtype=torch.int32, device="cuda")
        outs.append(dfv.moe_block_forward(L, x, ws, topk_idx=idx).clone())
        idxs.append(idx)
    dfv.set_path(True)
    assert torch.equal(idxs[0], idxs[1])
    a, b = outs[0].double(), outs[1].double()
    assert (a - b).abs().max().item() <= TOL_BF16 * b.abs().max().item()
    assert dfv.read_device_error(ws) == 0


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_fused_staging_modes_agree(dfv, a3b, mode):
    """Every gate/up staging mode of the single-launch kernel (row copies, 2-D
    tensor boxes, one 3-D box, one swizzled 3-D box with permuted MMA rows)
    computes the same output bit for bit, and each matches the oracle."""
    lw, ol, L = a3b
    x = hidden_without_near_ties(ol, 16, "bf16", seed=41)
    xg = x.cuda()
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    dfv.set_path(True)
    outs = {}
    try:
        for m in (3, mode):
            dfv.set_staging(m)
            outs[m] = dfv.moe_block_forward(L, xg, ws).clone()
            torch.cuda.synchronize()
            assert dfv.last_layer_path() == 1, dfv.fused_unavailable_reason()
            assert dfv.last_staging() <= m
    finally:
        dfv.set_staging(3)  # the library's default
    if mode > 0:
        assert dfv.last_staging() in (mode, mode - 1)
    assert torch.equal(outs[mode], outs[3])
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    assert _max_rel_err(_gpu_out_np(outs[mode]), ref) <= TOL_BF16


@pytest.fixture(scope="module")
def a3b_chain(dfv):
    """Six A3B-shape layers with distinct weights (7 GB, far larger than L2)."""
    lws = [inputs.make_layer(inputs.A3B, seed=900 + l, device="cuda") for l in range(6)]
    return lws, [dfv.Layer(w) for w in lws]


@pytest.mark.parametrize("k,mode", [(1, "independent"), (3, "repeated"), (8, "repeated"),
                                    (12, "independent"), (13, "repeated"), (16, "independent")])
def test_chained_launches_equal_isolated_launches(dfv, a3b_chain, k, mode):
    """Layer launches chained back to back must give, bit for bit, what the same
    launches give one at a time with a device synchronisation in between.
    Every output depends only on its own row and each launch's layer.  So any
    difference means a launch read data it should not have: a stage before its
    copy landed, a stage that was being refilled, or another launch's workspace.
    Covers eager chains and CUDA-graph replays, for ring sizes of both
    parities (k <= 8 and k > 8)."""
    _, Ls = a3b_chain
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x = inputs.make_hidden(k, 2048, "bf16", seed=4000 + k, mode=mode, device="cuda")
    iso = []
    for L in Ls:
        o = dfv.moe_block_forward(L, x, ws)
        torch.cuda.synchronize()
        iso.append(o.clone())
    assert dfv.last_layer_path() == 1, dfv.fused_unavailable_reason()
    outs = [torch.empty_like(x) for _ in Ls]

    def chain():
        for L, o in zip(Ls, outs):
            dfv.moe_block_forward(L, x, ws, out=o)

    for _ in range(40):
        chain()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(outs, iso))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(40):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(outs, iso))
    assert dfv.read_device_error(ws) == 0
