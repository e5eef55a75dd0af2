"""GPU parity of the mxfp4 expert path (E2M1 codes + one E8M0 scale per 32
elements, widened in registers) through the C ABI, against the CPU oracle,
which decodes every code exactly to fp64.

Routing is bit-exact as for bf16 (the router weights are bf16).  Outputs must
satisfy max|err| <= 5e-2 * max|ref|.  The weights and the bf16 inputs reach the
tensor cores exactly; the one rounding on the way is h = silu(g) * u, held
with 11 significant bits, so the observed error is far below that bar and a
tighter check (one-hot inputs, where every output is a short sum) pins the
decode of every code and scale."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import hidden_without_near_ties, np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

TOL_MXFP4 = 5e-2
# one-hot rows: y_r = sum_i h_i * Wd[r, i] with h_i carried in 11 bits; the
# error is <= 2^-12 * sum_i |h_i Wd[r, i]|, a few 1e-4 of max|y| for these sizes
TOL_DECODE = 4e-3


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


def _fused_ok(d, I):
    """Shapes the single-launch mxfp4 kernel takes (others use the multi-launch path)."""
    return d % 512 == 0 and d <= 2048 and I % 128 == 0 and 128 <= I <= 512


def _check_path(dfv, path, d=2048, I=512):
    want = 1 if (path == "fused" and _fused_ok(d, I)) else 0
    assert dfv.last_layer_path() == want, dfv.fused_unavailable_reason()


def _max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(got.astype(np.float64) - ref)) / max(scale, 1e-30))


def _out_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _bf16_np(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()


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


def _shape(d, E, K, I, scale_exp=(119, 127)):
    return inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype="mxfp4", scale_exp=scale_exp)


def _one_hot_rows(k, d, seed):
    g = torch.Generator().manual_seed(seed)
    cols = torch.randperm(d, generator=g)[:k]
    x = torch.zeros(k, d)
    x[torch.arange(k), cols] = 1.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d,I", [(64, 64), (128, 192), (320, 128), (512, 64), (512, 128), (1024, 192), (2048, 384),
                                 (2048, 448)])
@pytest.mark.parametrize("scale_exp", [(119, 127), (113, 140)])
def test_decode_every_code_and_scale_one_hot(dfv, path, d, I, scale_exp):
    """One expert, K = 1 (routing weight exactly 1): with one-hot rows the gate
    and up values are single weights, so a wrong nibble order, sign, code or
    scale shows up as an O(1) error.  Scales span the whole exact range."""
    s = _shape(d, 1, 1, I, scale_exp)
    lw = inputs.make_layer(s, seed=d + I)
    ol = oracle_layer(lw)
    k = 16
    x = _one_hot_rows(k, d, seed=d)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    out = dfv.moe_block_forward(L, x.cuda(), ws)
    torch.cuda.synchronize()
    _check_path(dfv, path, d, I)
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x))
    # compare per row (rows differ in magnitude by up to 2^36 with wide scales)
    got = _out_np(out)
    for t in range(k):
        assert _max_rel_err(got[t:t + 1], ref[t:t + 1]) <= TOL_DECODE, t


def _wide_scale_layer(d, I):
    """One expert, K = 1: gate scales drawn over 0..251 and each up scale 251
    minus its gate scale (g * u stays near 1, so h is finite and normal); each
    down row r has one scale s_r spread over 20..219."""
    s = _shape(d, 1, 1, I)
    lw = inputs.make_layer(s, seed=d + 3 * I)
    g = torch.Generator().manual_seed(d + I)
    lw.s_gate = torch.randint(0, 252, lw.s_gate.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    lw.s_up = (251 - lw.s_gate.to(torch.int32)).to(torch.uint8)
    srow = (20 + (torch.arange(d) * 37) % 200).to(torch.uint8)
    lw.s_down = srow.view(1, d, 1).expand(lw.s_down.shape).contiguous()
    assert int(lw.s_gate.min()) == 0 and int(lw.s_gate.max()) == 251
    return lw, srow


def _check_every_scale(dfv, lw, srow, d, I, fused):
    ol = oracle_layer(lw)
    k = 16
    x = _one_hot_rows(k, d, seed=d + 1)
    dfv.set_path(fused)
    try:
        L = dfv.Layer(lw.to("cuda"))
        ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
        out = dfv.moe_block_forward(L, x.cuda(), ws)
        torch.cuda.synchronize()
        _check_path(dfv, "fused" if fused else "multi", d, I)
    finally:
        dfv.set_path(True)
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x))
    norm = np.exp2(srow.double().numpy() - 127.0)
    got = _out_np(out) / norm
    refn = ref / norm
    assert np.all(np.isfinite(got))
    for t in range(k):
        assert _max_rel_err(got[t:t + 1], refn[t:t + 1]) <= TOL_DECODE, t


@pytest.mark.parametrize("d,I", [(512, 256), (2048, 512), (1024, 128)])
def test_fused_decode_exact_for_every_scale(dfv, d, I):
    """The single-launch kernel applies each block's scale to fp32 partial
    sums, so every E8M0 exponent is exact as long as the values stay inside
    the fp32 range (above 251 the largest E2M1 codes, 6 * 2^125, would leave
    it at any input).  With one-hot rows every output is a short sum; each
    output is divided by 2^(s_r - 127) before the comparison, so rows of every
    magnitude are held to the same bar."""
    lw, srow = _wide_scale_layer(d, I)
    _check_every_scale(dfv, lw, srow, d, I, fused=True)


@pytest.mark.parametrize("d,I", [(512, 256), (2048, 512), (320, 64), (1024, 192), (4096, 1536)])
def test_multi_launch_decode_exact_for_every_scale(dfv, d, I):
    """The multi-launch mxfp4 kernels also scale each 32-element block's fp32
    partial sum (a quad's lanes hold one block per MMA pair), so they are exact
    for every scale too and set no device error.  d = 320 and d_ff = 64 or 192
    end in half chunks of 64 codes; d = 4096 is wider than the single launch
    takes."""
    lw, srow = _wide_scale_layer(d, I)
    _check_every_scale(dfv, lw, srow, d, I, fused=False)


SMALL = [
    # d, E, K, I: d % 128 == 64 and d_ff % 128 == 64 exercise half chunks
    (320, 24, 3, 192),
    (512, 40, 8, 128),
    (256, 8, 8, 64),  # K == E: every row wakes every expert
    (512, 16, 4, 192),   # multi-launch path: ragged d_ff chunk
    (512, 16, 4, 256),   # single-launch kernel: one gate/up stage per unit, two 64-byte boxes per down row
    (2048, 24, 8, 128),  # single-launch kernel: four gate/up stages per unit
    (512, 8, 1, 128),    # top-1 routing, fewer experts than a warp has lanes
    (1024, 4, 2, 384),   # four experts: up to 16 tokens each (both token tiles), three boxes per down row
    (1024, 4, 2, 448),   # multi-launch path: up to 16 tokens per expert
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("k", [1, 3, 8, 9, 16])
def test_mxfp4_layer_parity_small(dfv, path, shape, k):
    d, E, K, I = shape
    lw = inputs.make_layer(_shape(d, E, K, I), seed=700 + k)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=800 + k)
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    _check_routing(dfv, L, ol, xg, ws)
    out = dfv.moe_block_forward(L, xg, ws)
    torch.cuda.synchronize()
    assert dfv.read_device_error(ws) == 0
    _check_path(dfv, path, d, I)
    ref = oracle.moe_forward(ol, np_of(x), nthreads=8)
    assert _max_rel_err(_out_np(out), ref) <= TOL_MXFP4


@pytest.fixture(scope="module")
def mx_full(dfv):
    lw = inputs.make_layer(inputs.MXFP4, seed=9, device="cuda")
    return lw, oracle_layer(lw.to("cpu")), dfv.Layer(lw)


@pytest.mark.parametrize("k,mode", [(1, "independent"), (16, "independent"), (16, "repeated"), (5, "independent")])
def test_mxfp4_full_size(dfv, mx_full, path, k, mode):
    """E=256, top-8, d=2048, d_ff=512 at the block sizes of decode and verify."""
    lw, ol, L = mx_full
    x = hidden_without_near_ties(ol, k, "bf16", seed=900 + k, mode=mode)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    W = _check_routing(dfv, L, ol, xg, ws)
    assert W <= min(256, 8 * k)
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, xg, ws, n_woken=nw)
    torch.cuda.synchronize()
    _check_path(dfv, path)
    assert int(nw.item()) == W
    assert dfv.read_device_error(ws) == 0
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    err = _max_rel_err(_out_np(out), ref)
    assert err <= TOL_MXFP4


def test_mxfp4_block_of_identical_rows(dfv, mx_full, path):
    """A block of k copies of one row wakes that row's K experts only, and every
    output row equals the single-row result."""
    lw, ol, L = mx_full
    x1 = inputs.make_hidden(1, 2048, "bf16", seed=21, device="cuda")
    x = x1.repeat(16, 1).contiguous()
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, x, ws, n_woken=nw).clone()
    torch.cuda.synchronize()
    assert int(nw.item()) == 8
    assert all(torch.equal(out[t], out[0]) for t in range(16))


def test_mxfp4_stack_teacher_forced(dfv, path):
    """Pre-norm residual stack of mxfp4 layers: each GPU layer checked against
    the oracle on the GPU's own layer input; one call over all layers equals the
    layer-by-layer calls bit for bit."""
    shape = _shape(512, 32, 4, 128)
    n_layers, k = 4, 16
    lws = [inputs.make_layer(shape, seed=950 + l, device="cuda") for l in range(n_layers)]
    Ls = [dfv.Layer(w) for w in lws]
    ols = [oracle_layer(w.to("cpu")) for w in lws]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16) for L in Ls))
    x0 = inputs.make_hidden(k, 512, "bf16", seed=951, device="cuda")
    x = x0.clone()
    excluded = 0
    for l in range(n_layers):
        xin = x.clone()
        dfv.moe_stack_forward([Ls[l]], x, ws)
        torch.cuda.synchronize()
        xin_np = np_of(xin)
        ref = oracle.stack_forward([ols[l]], xin_np)
        nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in oracle.rmsnorm(xin_np)], dtype=np.uint16)
        lg, _, _ = oracle.route(ols[l], nb)
        keep = topk_gap(lg, shape.top_k) >= 1e-3
        excluded += int((~keep).sum())
        got = _out_np(x)[keep]
        refd = _bf16_np(ref)[keep]
        delta_ref = refd - _out_np(xin)[keep]
        bound = TOL_MXFP4 * max(np.max(np.abs(delta_ref)), 1e-30) + np.max(np.abs(refd)) * 2 ** -8
        assert np.max(np.abs(got - refd)) <= bound, "layer %d" % l
    assert excluded <= n_layers * k // 4
    assert dfv.read_device_error(ws) == 0
    xs = x0.clone()
    dfv.moe_stack_forward(Ls, xs, ws)
    torch.cuda.synchronize()
    assert torch.equal(xs, x)


def test_mxfp4_block_rows_equal_single_token_calls_fused(dfv, mx_full):
    """Single-launch path: row t of a 16-row block is bit-identical to the k=1
    call on that row (every output's summation order depends only on its own
    token)."""
    lw, ol, L = mx_full
    dfv.set_path(True)
    x = inputs.make_hidden(16, 2048, "bf16", seed=31, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    blk = dfv.moe_block_forward(L, x, ws).clone()
    _check_path(dfv, "fused")
    for t in range(16):
        row = dfv.moe_block_forward(L, x[t:t + 1].contiguous(), ws)
        torch.cuda.synchronize()
        assert torch.equal(row[0], blk[t]), t
    assert dfv.read_device_error(ws) == 0


@pytest.mark.parametrize("shape", [(2048, 256, 8, 512), (1024, 16, 4, 256), (2560, 8, 2, 1024)])
def test_mxfp4_block_rows_equal_single_token_calls_multi_launch(dfv, shape):
    """Multi-launch path: row t of a 16-row block is bit-identical to the k=1
    call on that row.  The gate/up split of d is chosen for the largest block
    whatever k is, so every row's sums run in one order."""
    d, E, K, I = shape
    lw = inputs.make_layer(inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype="mxfp4"), seed=d + E,
                           device="cuda")
    L = dfv.Layer(lw)
    x = inputs.make_hidden(16, d, "bf16", seed=37, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    dfv.set_path(False)
    try:
        blk = dfv.moe_block_forward(L, x, ws).clone()
        _check_path(dfv, "multi")
        for t in (0, 7, 8, 15):
            row = dfv.moe_block_forward(L, x[t:t + 1].contiguous(), ws)
            torch.cuda.synchronize()
            assert torch.equal(row[0], blk[t]), t
    finally:
        dfv.set_path(True)
    assert dfv.read_device_error(ws) == 0


def test_mxfp4_fused_and_multikernel_paths_agree(dfv, mx_full):
    lw, ol, L = mx_full
    x = inputs.make_hidden(16, 2048, "bf16", seed=32, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    outs, idxs = [], []
    for fused in (True, False):
        dfv.set_path(fused)
        idx = torch.empty(16, 8, dtype=torch.int32, device="cuda")
        outs.append(dfv.moe_block_forward(L, x, ws, topk_idx=idx).clone())
        idxs.append(idx)
        _check_path(dfv, "fused" if fused else "multi")
    dfv.set_path(True)
    assert torch.equal(idxs[0], idxs[1])
    a, b = outs[0].double(), outs[1].double()
    assert (a - b).abs().max().item() <= TOL_MXFP4 * b.abs().max().item()
    assert dfv.read_device_error(ws) == 0


@pytest.fixture(scope="module")
def mx_chain(dfv):
    """Six mxfp4 layers with distinct weights (E=256, d=2048, d_ff=512)."""
    lws = [inputs.make_layer(inputs.MXFP4, seed=950 + l, device="cuda") for l in range(6)]
    return lws, [dfv.Layer(w) for w in lws]


@pytest.mark.parametrize("k,mode", [(1, "independent"), (5, "repeated"), (9, "repeated"), (16, "independent")])
def test_mxfp4_chained_launches_equal_isolated_launches(dfv, mx_chain, k, mode):
    """Back-to-back launches of the single-launch mxfp4 kernel (eager chains and
    CUDA-graph replays) give, bit for bit, what isolated launches give: every
    output depends only on its own row and its launch's layer."""
    _, Ls = mx_chain
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], 16))
    x = inputs.make_hidden(k, 2048, "bf16", seed=4100 + k, mode=mode, device="cuda")
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
