"""GPU parity of the 8-bit expert path through the C ABI, against the CPU
oracle.  "Speculating on a Strix Halo (part 2)", section "The verification
cog", runs the target "at Q8"; the pages fix no format, and the reading taken
is llama.cpp's Q8_0 block: 32 int8 codes of a row share one IEEE binary16
scale, value = code * scale.  The single-launch kernel widens each code to
fp16 exactly and applies the block's scale to the fp32 partial sum of that
block, so the only roundings are the fp32 sums and h = silu(g) * u held in
fp16 with 11 significant bits.

Routing is bit-exact (bf16 router).  Outputs: max|err| <= 2e-2 * max|ref|
(the bf16 bar: the weights reach the tensor cores exactly)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import hidden_without_near_ties, np_of, oracle_layer

pytestmark = pytest.mark.gpu

TOL_Q8 = 2e-2
TOL_DECODE = 4e-3


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    m.set_path(True)
    return m


def _shape(d, E, K, I, ns=0):
    return inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype="q8", n_shared=ns)


def _rel(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _run(dfv, lw, x, ws=None):
    L = dfv.Layer(lw.to("cuda"))
    if ws is None:
        ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    idx = torch.empty(x.shape[0], lw.shape.top_k, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, x.cuda(), ws, topk_idx=idx)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == 1, dfv.fused_unavailable_reason()
    assert dfv.read_device_error(ws) == 0
    return out.double().cpu().numpy(), idx.cpu().numpy()


SMALL = [
    # d, E, K, I
    (512, 32, 4, 128),    # one down stage of two 64-byte boxes
    (256, 16, 2, 64),     # one gate/up stage per unit, one box per down row
    (1024, 40, 8, 256),   # four gate/up stages, a full down stage
    (512, 8, 8, 512),     # K == E; two down stages per unit (scales by tensor map)
    (768, 4, 2, 192),     # up to 16 tokens per expert
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("k", [1, 3, 8, 9, 16])
def test_q8_layer_parity_small(dfv, shape, k):
    d, E, K, I = shape
    lw = inputs.make_layer(_shape(d, E, K, I), seed=1700 + k + d)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=1800 + k)
    out, idx = _run(dfv, lw, x)
    _, ridx, _ = oracle.route(ol, np_of(x))
    assert np.array_equal(idx, ridx)
    ref = oracle.moe_forward(ol, np_of(x), nthreads=8)
    assert _rel(out, ref) <= TOL_Q8


@pytest.mark.parametrize("k", [1, 16])
def test_q8_shared_expert(dfv, k):
    lw = inputs.make_layer(_shape(1024, 16, 4, 256, ns=1), seed=1900 + k)
    ol = oracle_layer(lw)
    x = hidden_without_near_ties(ol, k, "bf16", seed=1950 + k)
    out, _ = _run(dfv, lw, x)
    assert _rel(out, oracle.moe_forward(ol, np_of(x), nthreads=8)) <= TOL_Q8


@pytest.fixture(scope="module")
def q8_full(dfv):
    lw = inputs.make_layer(inputs.Q8, seed=19, device="cuda")
    return lw, oracle_layer(lw.to("cpu")), dfv.Layer(lw)


@pytest.mark.parametrize("k,mode", [(1, "independent"), (16, "independent"), (16, "repeated")])
def test_q8_full_size(dfv, q8_full, k, mode):
    """E=256, top-8, d=2048, d_ff=512, the mxfp4 configuration's shape."""
    lw, ol, L = q8_full
    x = hidden_without_near_ties(ol, k, "bf16", seed=2000 + k, mode=mode)
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    idx = torch.empty(k, 8, dtype=torch.int32, device="cuda")
    out = dfv.moe_block_forward(L, x.cuda(), ws, topk_idx=idx)
    torch.cuda.synchronize()
    assert dfv.last_layer_path() == 1
    assert dfv.read_device_error(ws) == 0
    _, ridx, _ = oracle.route(ol, np_of(x))
    assert np.array_equal(idx.cpu().numpy(), ridx)
    ref = oracle.moe_forward(ol, np_of(x), nthreads=oracle.num_threads_available())
    assert _rel(out.double().cpu().numpy(), ref) <= TOL_Q8


def _one_hot_rows(k, d, seed):
    g = torch.Generator().manual_seed(seed)
    cols = torch.randperm(d, generator=g)[:k]
    x = torch.zeros(k, d)
    x[torch.arange(k), cols] = 1.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d,I", [(256, 64), (512, 256), (2048, 512)])
def test_q8_decode_every_code_and_wide_scales_one_hot(dfv, d, I):
    """One expert, K = 1, one-hot rows, and a down projection that copies h
    (W_down[r, i] = 1 for r = i, scale 1): output r of row t is then
    h_r = silu(g_r) * u_r with g_r and u_r single codes times single scales,
    checked element by element.  Gate and up codes cover all of -128..127;
    gate scales are binary16 values of both signs from 2^-20 to 2^11,
    subnormals included, and each up scale is 2^-floor(e/2) for its gate
    scale's exponent e, so h stays finite and normal.  A wrong byte order,
    sign, code or block scale is an O(1) error somewhere (elements far below
    their row's largest are held to a floor: see below)."""
    assert d >= I
    s = _shape(d, 1, 1, I)
    lw = inputs.make_layer(s, seed=d + I)
    g = torch.Generator().manual_seed(d * 3 + I)
    lw.w_gate = torch.randint(-128, 128, lw.w_gate.shape, generator=g, dtype=torch.int32).to(torch.int8)
    lw.w_up = torch.randint(-128, 128, lw.w_up.shape, generator=g, dtype=torch.int32).to(torch.int8)
    e = torch.randint(-20, 11, lw.s_gate.shape, generator=g).double()
    mant = 1.0 + torch.rand(lw.s_gate.shape, generator=g, dtype=torch.float64)
    sign = torch.where(torch.rand(lw.s_gate.shape, generator=g) < 0.5, -1.0, 1.0).double()
    lw.s_gate = (sign * mant * torch.exp2(e)).to(torch.float16)
    lw.s_up = torch.exp2(-torch.floor(e / 2)).to(torch.float16)
    assert bool((lw.s_gate.abs() < 2.0 ** -14).any())  # subnormal binary16 scales occur
    assert torch.isfinite(lw.s_gate.float()).all() and torch.isfinite(lw.s_up.float()).all()
    wd = torch.zeros_like(lw.w_down)
    wd[0, torch.arange(I), torch.arange(I)] = 1
    lw.w_down = wd
    lw.s_down = torch.ones_like(lw.s_down)
    ol = oracle_layer(lw)
    k = 16
    x = _one_hot_rows(k, d, seed=d + 7)
    out, _ = _run(dfv, lw, x)
    ref = oracle.moe_forward(ol, np_of(x))
    assert np.all(out[:, I:] == 0.0)
    err = np.abs(out - ref)
    # h reaches the down MMA as fp16 scaled by one power of two per row (its
    # largest magnitude in [1, 2)): elements more than 2^24 below the row's
    # largest lose bits or flush to zero, hence the floor of 2^-23 of the row
    # maximum
    floor = 2.0 ** -23 * np.max(np.abs(ref), axis=1, keepdims=True)
    # element by element: the bf16 output rounds by up to 2^-8 of the value and
    # h carries 2^-12 from its fp16 staging, hence 5e-3
    assert np.all(err <= 5e-3 * np.abs(ref) + floor), float(np.max(err / (np.abs(ref) + floor)))


def test_q8_block_rows_equal_single_token_calls(dfv, q8_full):
    lw, ol, L = q8_full
    x = inputs.make_hidden(16, 2048, "bf16", seed=41, device="cuda")
    ws = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    blk = dfv.moe_block_forward(L, x, ws).clone()
    for t in range(16):
        row = dfv.moe_block_forward(L, x[t:t + 1].contiguous(), ws)
        torch.cuda.synchronize()
        assert torch.equal(row[0], blk[t]), t
    assert dfv.read_device_error(ws) == 0


def test_q8_unsupported_shape_and_path_are_refused(dfv):
    lw = inputs.make_layer(_shape(512, 8, 2, 384), seed=5)  # d_ff > 256 but not a multiple of 256
    L = dfv.Layer(lw.to("cuda"))
    ws = dfv.alloc_workspace(1 << 22)
    x = inputs.make_hidden(4, 512, "bf16", seed=6, device="cuda")
    with pytest.raises(dfv.DfvError) as ei:
        dfv.moe_block_forward(L, x, ws)
    assert ei.value.status == 2  # DFV_ERR_UNSUPPORTED
    lw2 = inputs.make_layer(_shape(512, 8, 2, 128), seed=5)
    L2 = dfv.Layer(lw2.to("cuda"))
    dfv.set_path(False)
    try:
        with pytest.raises(dfv.DfvError) as ei:
            dfv.moe_block_forward(L2, x, dfv.alloc_workspace(dfv.workspace_size(L2, 16)))
        assert ei.value.status == 2
    finally:
        dfv.set_path(True)


def test_q8_stack_teacher_forced(dfv):
    """Pre-norm residual stack of 8-bit layers: one call over four layers equals
    the layer-by-layer calls bit for bit, and each layer's MoE output matches
    the oracle on the GPU's own normalised input."""
    shape = _shape(512, 32, 4, 128)
    lws = [inputs.make_layer(shape, seed=2100 + l, device="cuda") for l in range(4)]
    Ls = [dfv.Layer(w) for w in lws]
    ws = dfv.alloc_workspace(max(dfv.workspace_size(L, 16) for L in Ls))
    x0 = inputs.make_hidden(16, 512, "bf16", seed=2199, device="cuda")
    x = x0.clone()
    for l in range(4):
        dfv.moe_stack_forward([Ls[l]], x, ws)
    torch.cuda.synchronize()
    xs = x0.clone()
    dfv.moe_stack_forward(Ls, xs, ws)
    torch.cuda.synchronize()
    assert torch.equal(xs, x)
    ref = oracle.stack_forward([oracle_layer(w.to("cpu")) for w in lws], np_of(x0))
    refd = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double()
    delta = (refd - x0.double().cpu()).abs().max().item()
    assert (x.double().cpu() - refd).abs().max().item() <= TOL_Q8 * 4 * delta + refd.abs().max().item() * 2 ** -7
    assert dfv.read_device_error(ws) == 0
