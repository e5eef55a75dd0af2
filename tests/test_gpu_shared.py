"""GPU parity of layers with an always-on shared expert ("Speculating on a
Strix Halo", section "What the pieces cost": the routed experts plus one
always-on shared expert; the model card it cites activates 8 routed plus 1
shared), through the C ABI, against the CPU oracle.

The shared expert is stored as expert index E and runs as one more woken
expert that every row selects with weight 1.  The caller's routing copies
describe the routed experts only and stay bit-exact; outputs are held to the
same bars as the routed-only layers (2e-2 * max|ref| for bf16 and fp32
weights, 5e-2 for mxfp4)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import hidden_without_near_ties, np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-2, "bf16": 2e-2, "mxfp4": 5e-2}


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    return m


@pytest.fixture(params=["fused", "multi"])
def path(request, dfv):
    dfv.set_path(request.param == "fused")
    yield request.param
    dfv.set_path(True)


def _rel(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _shape(d, E, K, I, w_dtype="bf16"):
    return inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype=w_dtype, n_shared=1)


def _routing_is_routed_only(dfv, L, ol, x, ws):
    """route_topk and the layer's optional copies describe the routed experts."""
    r = dfv.route_topk(L, x, ws)
    torch.cuda.synchronize()
    _, idx, _ = oracle.route(ol, np_of(x))
    wk, offs, gat = oracle.woken(idx, ol.n_experts)
    W = int(r["n_woken"].item())
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert W == len(wk)
    assert np.array_equal(r["woken"].cpu().numpy()[:W], wk)
    assert np.array_equal(r["offsets"].cpu().numpy()[:W + 1], offs)
    assert np.array_equal(r["gather"].cpu().numpy(), gat)
    return W


SMALL = [
    # d, E, K, I, dtype
    (352, 24, 3, 96, "bf16"),
    (512, 40, 8, 160, "bf16"),
    (256, 8, 8, 64, "bf16"),     # K == E: the shared expert follows every routed one
    (64, 4, 2, 32, "bf16"),
    (512, 16, 4, 192, "mxfp4"),
    (1024, 4, 2, 448, "mxfp4"),  # experts with up to 16 tokens, the shared one always
    (2048, 24, 8, 64, "mxfp4"),
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("k", [1, 8, 9, 16])
def test_shared_layer_parity_small(dfv, path, shape, k):
    d, E, K, I, wdt = shape
    lw = inputs.make_layer(_shape(d, E, K, I, wdt), seed=40 + k)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=50 + k)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    W = _routing_is_routed_only(dfv, L, ol, xg, ws)
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, xg, ws, n_woken=nw)
    torch.cuda.synchronize()
    assert int(nw.item()) == W
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=8)
    assert _rel(out, ref) <= TOL[wdt]
    # the shared term is really there: the routed-only oracle is far off
    ol.n_shared = 0
    assert _rel(out, oracle.moe_forward(ol, np_of(x), nthreads=8)) > 5 * TOL[wdt]


@pytest.mark.parametrize("k", [1, 4])
def test_shared_tiny_fp32(dfv, k):
    lw = inputs.make_layer(inputs.LayerShape(**{**inputs.TINY.__dict__, "n_shared": 1}), seed=3)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "f32", seed=4)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    out = dfv.moe_block_forward(L, x.cuda(), ws)
    torch.cuda.synchronize()
    assert _rel(out, oracle.moe_forward(ol, np_of(x))) <= TOL["f32"]


@pytest.fixture(scope="module")
def e256s(dfv):
    lw = inputs.make_layer(inputs.E256_SHARED, seed=17, device="cuda")
    return lw, oracle_layer(lw.to("cpu")), dfv.Layer(lw)


@pytest.mark.parametrize("k,mode", [(1, "independent"), (16, "independent"), (16, "repeated")])
def test_shared_full_size_sampled_rows(dfv, e256s, path, k, mode):
    """256 routed experts (top-8) + 1 shared, d=2048, d_ff=512, bf16, in the
    bench's launch configuration; the oracle checks three rows of the block
    (each row's output depends on that row alone)."""
    lw, ol, L = e256s
    x = hidden_without_near_ties(ol, k, "bf16", seed=60 + k, mode=mode)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    out = dfv.moe_block_forward(L, x.cuda(), ws)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == (1 if path == "fused" else 0), dfv.fused_unavailable_reason()
    assert dfv.read_device_error(ws) == 0
    for t in sorted({0, k // 2, k - 1}):
        ref = oracle.moe_forward(ol, np.ascontiguousarray(np_of(x)[t:t + 1]), nthreads=8)
        assert _rel(out[t:t + 1], ref) <= TOL["bf16"], "row %d" % t


def test_shared_block_rows_equal_single_token_calls(dfv, e256s, path):
    lw, ol, L = e256s
    x = inputs.make_hidden(16, 2048, "bf16", seed=61, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    blk = dfv.moe_block_forward(L, x, ws).clone()
    for t in (0, 5, 15):
        row = dfv.moe_block_forward(L, x[t:t + 1].contiguous(), ws)
        torch.cuda.synchronize()
        assert torch.equal(row[0], blk[t]), "row %d" % t


def test_shared_paths_agree_and_share_a_workspace_with_routed_layers(dfv, e256s):
    """Fused and multi-kernel paths compute the same function; a workspace
    sized for the shared layer also serves a routed-only layer in between."""
    lw, ol, L = e256s
    plain = inputs.make_layer(inputs.LayerShape(d=2048, n_experts=256, top_k=8, d_ff=512), seed=18, device="cuda")
    Lp = dfv.Layer(plain)
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16), dfv.workspace_size(Lp, 16)))
    x = inputs.make_hidden(16, 2048, "bf16", seed=62, device="cuda")
    a = dfv.moe_block_forward(L, x, ws).clone()
    dfv.moe_block_forward(Lp, x, ws)
    dfv.set_path(False)
    try:
        b = dfv.moe_block_forward(L, x, ws).clone()
    finally:
        dfv.set_path(True)
    torch.cuda.synchronize()
    assert dfv.read_device_error(ws) == 0
    rel = float((a.float() - b.float()).abs().max() / a.float().abs().max())
    assert rel <= 2e-2


def test_shared_stack_teacher_forced(dfv, path):
    """Pre-norm residual stack of shared-expert layers: each GPU layer against
    the oracle on the GPU's own layer input."""
    shape = _shape(512, 32, 4, 128)
    n_layers, k = 4, 16
    lws = [inputs.make_layer(shape, seed=70 + l, device="cuda") for l in range(n_layers)]
    Ls = [dfv.Layer(w) for w in lws]
    ols = [oracle_layer(w.to("cpu")) for w in lws]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16) for L in Ls))
    x0 = inputs.make_hidden(k, 512, "bf16", seed=71, device="cuda")
    x = x0.clone()
    for l in range(n_layers):
        xin = x.clone()
        dfv.moe_stack_forward([Ls[l]], x, ws)
        torch.cuda.synchronize()
        xin_np = np_of(xin)
        ref = oracle.stack_forward([ols[l]], xin_np)
        nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in oracle.rmsnorm(xin_np)], dtype=np.uint16)
        lg, _, _ = oracle.route(ols[l], nb)
        keep = topk_gap(lg, shape.top_k) >= 1e-3
        got = x.float().cpu().numpy().astype(np.float64)[keep]
        refd = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy()[keep]
        delta_ref = refd - xin.float().cpu().numpy().astype(np.float64)[keep]
        bound = TOL["bf16"] * max(np.max(np.abs(delta_ref)), 1e-30) + np.max(np.abs(refd)) * 2 ** -8
        assert np.max(np.abs(got - refd)) <= bound, "layer %d" % l
    xs = x0.clone()
    dfv.moe_stack_forward(Ls, xs, ws)
    torch.cuda.synchronize()
    assert torch.equal(xs, x)
    assert dfv.read_device_error(ws) == 0
