"""Batched verify through the C ABI: n_blocks verify blocks of k positions
(the MI355X / vLLM write-up, section "Results: Throughput and Speedup": up to
32 concurrent requests) through one bf16 MoE layer, the expert contractions on
the fifth-generation tensor cores.

Every row routes on its own, so the oracle's output for the batch is its
output row by row.  Routing (top-K experts) must equal the oracle's exactly on
rows drawn without near-ties, and equal the single-block path's on every row;
outputs within 2e-2 * max|ref| (bf16 weights, fp32 accumulation, h in bf16)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import np_of, oracle_layer, topk_gap

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def dfv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv as m
    m.set_path(True)
    return m


def rows_without_near_ties(ol, T, seed, mode="independent", k=16):
    """T bf16 rows; any row whose K-th and (K+1)-th router logits (oracle, fp32)
    lie within 1e-3 is redrawn on its own."""
    x = inputs.make_hidden(T, ol.d, "bf16", seed, mode=mode)
    for attempt in range(1, 50):
        lg, _, _ = oracle.route(ol, np_of(x))
        bad = np.nonzero(topk_gap(lg, ol.top_k) < 1e-3)[0]
        if len(bad) == 0:
            return x
        x[bad] = inputs.make_hidden(len(bad), ol.d, "bf16", seed * 100 + attempt)
    raise RuntimeError("near-ties persist")


def _run(dfv, L, x, n_blocks, ws=None):
    T = x.shape[0]
    if ws is None:
        ws = dfv.alloc_workspace(dfv.batch_workspace_size(L, T))
    idx = torch.empty(T, L.shape.top_k, dtype=torch.int32, device="cuda")
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dfv.moe_batch_forward(L, x.cuda(), n_blocks, ws, topk_idx=idx, n_woken=nw)
    torch.cuda.synchronize()
    assert dfv.read_device_error(ws) == 0
    return out, idx.cpu().numpy(), int(nw.item())


def _rel(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.parametrize("n_blocks,k", [(1, 16), (4, 16), (8, 7), (3, 1), (32, 2)])
@pytest.mark.parametrize("ns", [0, 1])
def test_batch_parity_small(dfv, n_blocks, k, ns):
    shape = inputs.LayerShape(d=256, n_experts=16, top_k=4, d_ff=128, n_shared=ns)
    lw = inputs.make_layer(shape, seed=600 + n_blocks + ns)
    ol = oracle_layer(lw)
    x = rows_without_near_ties(ol, n_blocks * k, seed=601 + k)
    L = dfv.Layer(lw.to("cuda"))
    out, idx, nw = _run(dfv, L, x, n_blocks)
    _, ridx, _ = oracle.route(ol, np_of(x))
    assert np.array_equal(idx, ridx)
    assert nw == len(np.unique(ridx))
    ref = oracle.moe_forward(ol, np_of(x), nthreads=8)
    assert _rel(out.double().cpu().numpy(), ref) <= TOL


@pytest.fixture(scope="module")
def a3b(dfv):
    lw = inputs.make_layer(inputs.A3B, seed=77, device="cuda")
    return lw, oracle_layer(lw.to("cpu")), dfv.Layer(lw)


@pytest.mark.parametrize("n_blocks", [1, 4, 32])
def test_batch_a3b_against_oracle_and_single_blocks(dfv, a3b, n_blocks):
    """Qwen3-A3B-like layer, k = 16: routing equal to the oracle's and to the
    single-block path's; outputs against the oracle on a sample of rows (every
    row of a small batch) and against the single-block path on every row."""
    lw, ol, L = a3b
    k, T = 16, 16 * n_blocks
    x = rows_without_near_ties(ol, T, seed=700 + n_blocks)
    out, idx, nw = _run(dfv, L, x, n_blocks)
    _, ridx, _ = oracle.route(ol, np_of(x))
    assert np.array_equal(idx, ridx)
    assert nw == len(np.unique(ridx))
    sample = np.arange(T) if T <= 64 else np.random.default_rng(n_blocks).choice(T, 48, replace=False)
    ref = oracle.moe_forward(ol, np.ascontiguousarray(np_of(x)[sample]), nthreads=oracle.num_threads_available())
    assert _rel(out.double().cpu().numpy()[sample], ref) <= TOL
    # the single-block path, block by block
    ws1 = dfv.alloc_workspace(dfv.workspace_size(L, 16))
    xg = x.cuda()
    for b in range(n_blocks):
        i1 = torch.empty(k, 8, dtype=torch.int32, device="cuda")
        o1 = dfv.moe_block_forward(L, xg[b * k:(b + 1) * k].contiguous(), ws1, topk_idx=i1)
        torch.cuda.synchronize()
        assert np.array_equal(i1.cpu().numpy(), idx[b * k:(b + 1) * k])
        a, r = out[b * k:(b + 1) * k].double(), o1.double()
        assert (a - r).abs().max().item() <= TOL * r.abs().max().item()


def test_batch_repeated_blocks_and_more_than_128_tokens_per_expert(dfv):
    """32 blocks of one repeated row each at top-1 over 4 experts: experts get
    more than 128 tokens (up to 512), so their units run in several passes."""
    shape = inputs.LayerShape(d=256, n_experts=4, top_k=1, d_ff=128)
    lw = inputs.make_layer(shape, seed=808)
    ol = oracle_layer(lw)
    base = rows_without_near_ties(ol, 2, seed=809)
    x = base.repeat(256, 1).contiguous()  # 512 rows, two distinct
    L = dfv.Layer(lw.to("cuda"))
    out, idx, nw = _run(dfv, L, x, 32)
    ref = oracle.moe_forward(ol, np_of(base))
    got = out.double().cpu().numpy()
    assert _rel(got[0::2], np.repeat(ref[0:1], 256, axis=0)) <= TOL
    assert _rel(got[1::2], np.repeat(ref[1:2], 256, axis=0)) <= TOL
    assert nw <= 2


def test_batch_rejects_bad_arguments(dfv, a3b):
    _, _, L = a3b
    x = torch.zeros(32, 2048, dtype=torch.bfloat16, device="cuda")
    ws = dfv.alloc_workspace(dfv.batch_workspace_size(L, 32))
    with pytest.raises(ValueError):
        dfv.moe_batch_forward(L, x, 3, ws)  # rows not in equal blocks (binding check)
    lib = dfv.lib()
    import ctypes
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.dfv_moe_batch_forward(L.ref, ctypes.c_void_p(x.data_ptr()), 33, 16, ctypes.c_void_p(x.data_ptr()),
                                     None, None, ctypes.c_void_p(ws.data_ptr()), ws.numel(), s) == 1
    assert lib.dfv_moe_batch_forward(L.ref, ctypes.c_void_p(x.data_ptr()), 2, 16, ctypes.c_void_p(x.data_ptr()),
                                     None, None, ctypes.c_void_p(ws.data_ptr()), 256, s) == 3
