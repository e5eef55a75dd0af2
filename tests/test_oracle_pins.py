"""Pins of the CPU oracle against facts fixed outside the oracle itself:
format definitions, library routines in special cases, closed forms, brute
force on tiny inputs and invariants of the method ("Speculating on a Strix
Halo", sections "Speculative decoding" and "What the pieces cost"; part 2,
sections "The verification cog" and "Why drafter performance doesn't really
matter").  CPU only."""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from speculative_decoding_moe_gb300 import inputs
from tests._util import np_of, oracle_layer, topk_gap

# ---------------------------------------------------------------- number formats


def test_bf16_widening_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    same = (got == r) | (np.isnan(got) & np.isnan(r))
    assert same.all()


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    # random finite float32 patterns over the whole exponent range, plus exact ties
    pats = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = pats.view(np.float32)
    f = f[np.isfinite(f)]
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, -ties, np.float32([0.0, -0.0, 1e-45, 3.0e38])])
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _e2m1_from_bits(code: int) -> float:
    """OCP MX element type E2M1 from its bit fields: sign(1) exponent(2, bias 1)
    mantissa(1); exponent 0 is subnormal (0.m x 2^0)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def test_e2m1_all_codes():
    for c in range(16):
        assert oracle.e2m1_value(c) == _e2m1_from_bits(c)
        assert math.copysign(1.0, oracle.e2m1_value(c)) == (-1.0 if c & 8 else 1.0)


def test_e8m0_all_exponents():
    for e in range(255):
        assert oracle.e8m0_value(e) == math.ldexp(1.0, e - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_mxfp4_decode_packing_and_scales_exhaustive():
    # one row per (code pair, scale): every code at an even and an odd column
    scales_e = list(range(119, 128))
    codes = np.arange(16, dtype=np.uint8)
    for e in scales_e:
        # 32 columns: column c holds code c % 16
        row_codes = np.array([codes[c % 16] for c in range(32)], dtype=np.uint8)
        packed = (row_codes[0::2] | (row_codes[1::2] << 4)).astype(np.uint8).reshape(1, 16)
        sc = np.array([[e]], dtype=np.uint8)
        got = oracle.decode_rows(oracle.MXFP4, packed, sc, 0, 1, 32)[0]
        want = np.array([_e2m1_from_bits(c % 16) * 2.0 ** (e - 127) for c in range(32)])
        assert np.array_equal(got, want)
    # low nibble is the even column
    packed = np.array([[0x2F] + [0] * 15], dtype=np.uint8)
    got = oracle.decode_rows(oracle.MXFP4, packed, np.array([[128]], dtype=np.uint8), 0, 1, 32)[0]
    assert got[0] == -12.0 and got[1] == 2.0


def test_fp16_widening_matches_numpy_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    assert math.copysign(1.0, oracle.fp16_to_double(0x8000)) == -1.0


def test_q8_decode_codes_and_scales_exhaustive():
    # 8-bit weights read as llama.cpp's Q8_0 block: 32 int8 codes of a row share
    # one binary16 scale.  Row r holds all 256 codes in 8 blocks, each with its
    # own scale (subnormal, negative, large), so a wrong block index or a code
    # read unsigned shows
    scale_bits = np.array([0x3C00, 0x0001, 0x03FF, 0xB800, 0x7BFF, 0x1A3D, 0x2E66, 0x0400], dtype=np.uint16)
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(1, 256)
    for shift in range(8):  # rotate the scales over the blocks
        sc = np.roll(scale_bits, shift).reshape(1, 8).view(np.float16)
        got = oracle.decode_rows(oracle.Q8, codes, sc, 0, 1, 256)[0]
        want = codes[0].astype(np.float64) * np.repeat(sc[0].astype(np.float64), 32)
        assert np.array_equal(got, want)


def test_q8_layer_equals_the_bf16_layer_of_the_same_values():
    # codes times a per-block power of two (2^-7 .. 2^-9) are exact in bf16, so
    # the q8 layer and the bf16 layer holding the decoded values must agree
    # exactly: this ties the q8 layout (rows, blocks along a row, the down
    # matrix's transposed shape) to the already-pinned bf16 path
    d, E, K, I = 128, 6, 2, 64
    g = torch.Generator().manual_seed(21)

    def pair(rows, cols):
        q = torch.randint(-127, 128, (E, rows, cols), generator=g, dtype=torch.int32).to(torch.int8)
        ex = torch.randint(7, 10, (E, rows, cols // 32), generator=g)
        sc = torch.pow(2.0, -ex.double()).to(torch.float16)
        val = q.double() * sc.double().repeat_interleave(32, dim=2)
        return q, sc, val.to(torch.bfloat16)

    (qg, sg, vg), (qu, su, vu), (qd, sd, vd) = pair(I, d), pair(I, d), pair(d, I)
    assert torch.equal(vg.double(), qg.double() * sg.double().repeat_interleave(32, dim=2))
    wr = (torch.randn(E, d, generator=g) * 0.05).to(torch.bfloat16)
    s8 = inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype="q8")
    s16 = inputs.LayerShape(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype="bf16")
    l8 = oracle_layer(inputs.LayerWeights(s8, wr, qg, qu, qd, sg, su, sd))
    l16 = oracle_layer(inputs.LayerWeights(s16, wr, vg, vu, vd))
    x = np_of(inputs.make_hidden(5, d, "bf16", seed=22))
    a, b = oracle.moe_forward(l8, x), oracle.moe_forward(l16, x)
    assert np.array_equal(a, b) and np.abs(a).max() > 0


def test_silu_closed_forms():
    # logistic(ln 3) = 3/4, logistic(-ln 3) = 1/4
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert oracle.silu(-math.log(3.0)) == pytest.approx(-0.25 * math.log(3.0), rel=1e-15)
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)


# ---------------------------------------------------------------- routing


def _tiny_layer(seed=0, **kw):
    shape = inputs.LayerShape(**{**inputs.TINY.__dict__, **kw})
    return inputs.make_layer(shape, seed)


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_brute_force_over_all_subsets(seed):
    lw = _tiny_layer(seed)
    ol = oracle_layer(lw)
    x = inputs.make_hidden(4, 256, "f32", seed)
    logits, idx, _ = oracle.route(ol, np_of(x))
    K, E = ol.top_k, ol.n_experts
    for t in range(4):
        lg = logits[t].astype(np.float64)
        best = None
        for sub in itertools.combinations(range(E), K):
            key = (sum(lg[list(sub)]), tuple(-i for i in sub))
            if best is None or key > best[0]:
                best = (key, sub)
        chosen = sorted(best[1], key=lambda e: (-lg[e], e))
        assert list(idx[t]) == chosen


def test_topk_ties_go_to_lowest_index():
    lw = _tiny_layer(1)
    wr = lw.w_router.clone()
    wr[9] = wr[3]          # experts 3 and 9 get bit-identical logits
    wr[12] = wr[3]
    lw.w_router = wr
    ol = oracle_layer(lw)
    x = inputs.make_hidden(4, 256, "f32", 1)
    # make expert 3's logit the row maximum by construction
    xs = np_of(x).copy()
    for t in range(4):
        xs[t] = np.sign(np_of(wr)[3]).astype(np.float32)
    logits, idx, _ = oracle.route(ol, xs)
    for t in range(4):
        assert logits[t, 3] == logits[t, 9] == logits[t, 12]
        assert list(idx[t]) == [3, 9]


def test_routing_weights_full_softmax_when_K_equals_E():
    lw = _tiny_layer(2, top_k=16)
    ol = oracle_layer(lw)
    x = inputs.make_hidden(3, 256, "f32", 2)
    logits, idx, w = oracle.route(ol, np_of(x))
    for t in range(3):
        p = softmax(logits[t].astype(np.float64))
        assert np.allclose(w[t], p[idx[t]], rtol=1e-13, atol=0)
        assert list(idx[t]) == sorted(range(16), key=lambda e: (-logits[t, e], e))


def test_routing_weights_unnormalised_are_softmax_probabilities():
    lw = _tiny_layer(3)
    ol = oracle_layer(lw)
    ol.norm_topk = 0
    x = inputs.make_hidden(4, 256, "f32", 3)
    logits, idx, w = oracle.route(ol, np_of(x))
    for t in range(4):
        p = softmax(logits[t].astype(np.float64))
        assert np.allclose(w[t], p[idx[t]], rtol=1e-13, atol=0)


def test_renormalised_weights_sum_to_one_and_descend():
    lw = _tiny_layer(4)
    ol = oracle_layer(lw)
    x = inputs.make_hidden(4, 256, "f32", 4)
    _, idx, w = oracle.route(ol, np_of(x))
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_router_logits_match_float64_matmul_for_bf16_inputs():
    shape = inputs.LayerShape(d=128, n_experts=8, top_k=2, d_ff=64)
    lw = inputs.make_layer(shape, 5)
    ol = oracle_layer(lw)
    x = inputs.make_hidden(3, 128, "bf16", 5)
    logits, _, _ = oracle.route(ol, np_of(x))
    ref = (x.double() @ lw.w_router.double().T).float().numpy()
    assert np.allclose(logits, ref, rtol=0, atol=1e-6)


# ---------------------------------------------------------------- woken union


def _brute_union(idx, E):
    k, K = idx.shape
    wk = sorted({int(e) for e in idx.ravel()})
    offs = [0]
    gather = []
    for e in wk:
        for t in range(k):
            for s in range(K):
                if idx[t, s] == e:
                    gather.append(t * K + s)
        offs.append(len(gather))
    return wk, offs, gather


@pytest.mark.parametrize("seed", range(5))
def test_woken_union_matches_set_brute_force(seed):
    rng = np.random.default_rng(seed)
    E, K, k = 24, 3, 7
    idx = np.stack([rng.choice(E, size=K, replace=False) for _ in range(k)]).astype(np.int32)
    wk, offs, gat = oracle.woken(idx, E)
    bw, bo, bg = _brute_union(idx, E)
    assert list(wk) == bw and list(offs) == bo and list(gat) == bg


def test_woken_invariants_on_router_output():
    lw = _tiny_layer(6)
    ol = oracle_layer(lw)
    E, K = ol.n_experts, ol.top_k
    for k in (1, 2, 4, 8):
        x = inputs.make_hidden(k, 256, "f32", 60 + k)
        _, idx, _ = oracle.route(ol, np_of(x))
        wk, offs, gat = oracle.woken(idx, E)
        W = len(wk)
        if k == 1:
            assert W == K
        assert W <= min(E, k * K)
        assert offs[-1] == k * K and np.all(np.diff(offs) >= 1)
        assert sorted(gat) == list(range(k * K))
    # identical rows wake identical sets: a block of one repeated row wakes K
    x = inputs.make_hidden(1, 256, "f32", 7).repeat(5, 1)
    _, idx, _ = oracle.route(ol, np_of(x))
    wk, offs, _ = oracle.woken(idx, E)
    assert len(wk) == K and list(np.diff(offs)) == [5] * K


# ---------------------------------------------------------------- expert FFN


def _manual_layer(d, I, E, wg, wu, wd, wr=None, K=1):
    f = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if wr is None:
        wr = np.zeros((E, d), dtype=np.float32)
    return oracle.Layer(d=d, n_experts=E, top_k=K, d_ff=I, w_dtype=oracle.F32, r_dtype=oracle.F32,
                        w_router=f(wr), w_gate=f(wg), w_up=f(wu), w_down=f(wd))


def test_swiglu_expert_closed_form_2x2():
    # x = (1, 0); gate rows give g = (ln 3, 0); up rows give u = (c, 7); Wd swaps.
    # h = (silu(ln 3) c, silu(0) 7) = (0.75 ln3 c, 0); y = Wd h = (0, 0.75 ln3 c)
    c = 1.25
    ln3 = float(np.float32(math.log(3.0)))  # the weight as stored (fp32)
    wg = [[[ln3, 5.0], [0.0, -2.0]]]
    wu = [[[c, 3.0], [7.0, 1.0]]]
    wd = [[[0.0, 1.0], [1.0, 0.0]]]
    L = _manual_layer(2, 2, 1, wg, wu, wd)
    y = oracle.expert_ffn(L, 0, np.array([1.0, 0.0]))
    want = ln3 / (1.0 + 1.0 / 3.0 * math.exp(math.log(3.0) - ln3)) * c
    assert y[0] == 0.0
    assert y[1] == pytest.approx(want, rel=1e-15)
    assert y[1] == pytest.approx(0.75 * math.log(3.0) * c, rel=1e-7)


def test_swiglu_expert_rectangular_indexing():
    # d=3, I=2: only Wg[1,2], Wu[1,2] and Wd[0,1] are non-zero, so a transposed
    # or mis-strided operand lands on a zero.
    d, I = 3, 2
    wg = np.zeros((1, I, d)); wg[0, 1, 2] = math.log(3.0)
    wu = np.zeros((1, I, d)); wu[0, 1, 2] = 2.0
    wd = np.zeros((1, d, I)); wd[0, 0, 1] = -4.0
    L = _manual_layer(d, I, 1, wg, wu, wd)
    y = oracle.expert_ffn(L, 0, np.array([0.0, 0.0, 1.0]))
    g = float(np.float32(math.log(3.0)))
    want = -4.0 * (g / (1.0 + math.exp(-g))) * 2.0
    assert y[1] == 0.0 and y[2] == 0.0
    assert y[0] == pytest.approx(want, rel=1e-15)


def test_ffn_is_linear_in_down_weights_and_zero_with_zero_gate():
    lw = _tiny_layer(8)
    ol = oracle_layer(lw)
    x = np.random.default_rng(8).standard_normal(256)
    y = oracle.expert_ffn(ol, 3, x)
    lw2 = inputs.LayerWeights(lw.shape, lw.w_router, lw.w_gate, lw.w_up, lw.w_down * 2)
    y2 = oracle.expert_ffn(oracle_layer(lw2), 3, x)
    assert np.array_equal(y2, 2 * y)
    lw3 = inputs.LayerWeights(lw.shape, lw.w_router, torch.zeros_like(lw.w_gate), lw.w_up, lw.w_down)
    assert np.all(oracle.expert_ffn(oracle_layer(lw3), 3, x) == 0)


def test_identical_experts_make_routing_irrelevant():
    lw = _tiny_layer(9)
    same = lambda t: t[:1].expand_as(t).contiguous()
    lw = inputs.LayerWeights(lw.shape, lw.w_router, same(lw.w_gate), same(lw.w_up), same(lw.w_down))
    ol = oracle_layer(lw)
    x = inputs.make_hidden(4, 256, "f32", 9)
    out = oracle.moe_forward(ol, np_of(x))
    for t in range(4):
        y = oracle.expert_ffn(ol, 0, np_of(x)[t].astype(np.float64))
        assert np.allclose(out[t], y, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- shared expert
# "What the pieces cost": one always-on shared expert next to the routed ones
# (the cited model card: 8 routed plus 1 shared activated).  Reading: same
# SwiGLU form and size, applied to every row, weight 1, stored as expert E.


def test_shared_expert_closed_form_at_index_E():
    # two routed experts with zero weights (routed sum exactly 0) and a shared
    # expert (index 2) with one non-zero entry per matrix: a shared expert
    # read from another index, or transposed, gives zeros
    d, I, E = 3, 2, 2
    wg = np.zeros((E + 1, I, d)); wg[2, 1, 2] = math.log(3.0)
    wu = np.zeros((E + 1, I, d)); wu[2, 1, 2] = 2.0
    wd = np.zeros((E + 1, d, I)); wd[2, 0, 1] = -4.0
    L = _manual_layer(d, I, E, wg, wu, wd)
    L.n_shared = 1
    x = np.array([[0.0, 0.0, 1.0], [0.0, 0.0, -2.0]], dtype=np.float32)
    out = oracle.moe_forward(L, x)
    g = float(np.float32(math.log(3.0)))
    for t, xt in enumerate((1.0, -2.0)):
        z = g * xt
        want = -4.0 * (z / (1.0 + math.exp(-z))) * (2.0 * xt)
        assert out[t, 1] == 0.0 and out[t, 2] == 0.0
        assert out[t, 0] == pytest.approx(want, rel=1e-15)
    L.n_shared = 0
    assert np.all(oracle.moe_forward(L, x) == 0.0)


@pytest.mark.parametrize("j", [0, 7, 15])
def test_shared_copy_of_the_chosen_expert_doubles_the_output(j):
    # top-1 with renormalised weights gives the chosen expert weight exactly 1;
    # a router that sends every row to expert j and a shared expert holding a
    # copy of j's weights must give exactly twice the routed output
    lw = _tiny_layer(12, n_shared=1, top_k=1)
    wr = torch.zeros_like(lw.w_router)
    wr[j] = 1.0
    wg, wu, wd = lw.w_gate.clone(), lw.w_up.clone(), lw.w_down.clone()
    wg[-1], wu[-1], wd[-1] = wg[j], wu[j], wd[j]
    lw = inputs.LayerWeights(lw.shape, wr, wg, wu, wd)
    x = np_of(inputs.make_hidden(4, 256, "f32", 12).abs())  # logit of j = sum |x| > 0 = the others
    ol = oracle_layer(lw)
    _, idx, w = oracle.route(ol, x)
    assert np.all(idx == j) and np.all(w == 1.0)
    both = oracle.moe_forward(ol, x)
    ol.n_shared = 0
    routed = oracle.moe_forward(ol, x)
    assert np.array_equal(both, 2.0 * routed)
    assert not np.array_equal(both, routed)


def test_shared_expert_is_independent_of_routing():
    # relabelling the routed experts (router rows and weights together) leaves
    # the output unchanged; the shared expert stays last
    lw = _tiny_layer(13, n_shared=1)
    perm = torch.cat([torch.randperm(16, generator=torch.Generator().manual_seed(13)), torch.tensor([16])])
    lp = inputs.LayerWeights(lw.shape, lw.w_router[perm[:16]].contiguous(), lw.w_gate[perm].contiguous(),
                             lw.w_up[perm].contiguous(), lw.w_down[perm].contiguous())
    x = np_of(inputs.make_hidden(4, 256, "f32", 13))
    a = oracle.moe_forward(oracle_layer(lw), x)
    b = oracle.moe_forward(oracle_layer(lp), x)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-16)
    # and the shared term is the same whatever the router does
    lz = inputs.LayerWeights(lw.shape, torch.zeros_like(lw.w_router), lw.w_gate, lw.w_up, lw.w_down)
    lr = inputs.LayerWeights(lw.shape, lw.w_router, lw.w_gate, lw.w_up, lw.w_down)
    dz = oracle.moe_forward(oracle_layer(lz), x)
    dr = oracle.moe_forward(oracle_layer(lr), x)
    olz, olr = oracle_layer(lz), oracle_layer(lr)
    olz.n_shared = olr.n_shared = 0
    assert np.allclose(dz - oracle.moe_forward(olz, x), dr - oracle.moe_forward(olr, x), rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- block invariants


@pytest.mark.parametrize("n_shared", [0, 1])
@pytest.mark.parametrize("w_dtype", ["f32", "bf16", "mxfp4", "q8"])
def test_block_equals_row_by_row_decode(w_dtype, n_shared):
    shape = inputs.LayerShape(d=128, n_experts=12, top_k=3, d_ff=64, w_dtype=w_dtype,
                              r_dtype="f32" if w_dtype == "f32" else "bf16",
                              act="f32" if w_dtype == "f32" else "bf16", n_shared=n_shared)
    lw = inputs.make_layer(shape, 10)
    ol = oracle_layer(lw)
    x = np_of(inputs.make_hidden(6, 128, shape.act, 10))
    blk = oracle.moe_forward(ol, x)
    for t in range(6):
        row = oracle.moe_forward(ol, np.ascontiguousarray(x[t:t + 1]))
        assert np.array_equal(row[0], blk[t])


def test_expert_relabelling_does_not_change_output():
    lw = _tiny_layer(11)
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(11))
    lp = inputs.LayerWeights(lw.shape, lw.w_router[perm].contiguous(), lw.w_gate[perm].contiguous(),
                             lw.w_up[perm].contiguous(), lw.w_down[perm].contiguous())
    x = np_of(inputs.make_hidden(4, 256, "f32", 11))
    a = oracle.moe_forward(oracle_layer(lw), x)
    b = oracle.moe_forward(oracle_layer(lp), x)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-16)


def test_rmsnorm_closed_forms():
    x = np.array([[3.0, 4.0], [-2.0, -2.0]], dtype=np.float32)
    y = oracle.rmsnorm(x, eps=1e-6)
    assert y[0] == pytest.approx(np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-6), rel=1e-15)
    assert y[1] == pytest.approx(-1.0 / math.sqrt(1.0 + 1e-6 / 4.0) * np.ones(2), rel=1e-15)


def test_stack_with_zero_down_weights_is_identity():
    shape = inputs.LayerShape(d=128, n_experts=8, top_k=2, d_ff=64)
    layers = []
    for s in range(3):
        lw = inputs.make_layer(shape, 20 + s)
        lw.w_down = torch.zeros_like(lw.w_down)
        layers.append(oracle_layer(lw))
    x = np_of(inputs.make_hidden(5, 128, "bf16", 20))
    assert np.array_equal(oracle.stack_forward(layers, x), x)


def test_stack_one_layer_is_prenorm_residual():
    shape = inputs.LayerShape(d=128, n_experts=8, top_k=2, d_ff=64)
    ol = oracle_layer(inputs.make_layer(shape, 30))
    x = np_of(inputs.make_hidden(5, 128, "bf16", 30))
    got = oracle.stack_forward([ol], x)
    n = oracle.rmsnorm(x)
    nb = np.array([[oracle.double_to_bf16(v) for v in r] for r in n], dtype=np.uint16)
    moe = oracle.moe_forward(ol, nb)
    xd = np.vectorize(oracle.bf16_to_double)(x)
    want = np.array([[oracle.double_to_bf16(v) for v in r] for r in xd + moe], dtype=np.uint16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- acceptance


def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(12)
    lg = rng.standard_normal((7, 1000)).astype(np.float32)
    lg[2, [10, 500]] = 9.0                  # tie: lowest index wins
    lg[3, :] = 0.0
    lg[3, 999] = -0.0
    lg[4, [0, 1]] = [0.0, -0.0]             # +0 and -0 are equal
    lg[4, 2:] = -1.0
    got = oracle.argmax_rows(lg)
    assert list(got) == list(np.argmax(lg, axis=1))
    b = torch.from_numpy(lg).to(torch.bfloat16)
    assert list(oracle.argmax_rows(np_of(b))) == list(np.argmax(b.float().numpy(), axis=1))


@pytest.mark.parametrize("k", [0, 1, 4, 15, 16])
def test_accept_is_longest_matching_prefix_plus_one(k):
    rng = np.random.default_rng(13 + k)
    lg = rng.standard_normal((k + 1, 300)).astype(np.float32)
    a = np.argmax(lg, axis=1)
    for n in range(k + 1):
        draft = rng.integers(0, 300, size=k).astype(np.int32)
        draft[:n] = a[:n]
        if n < k:
            draft[n] = (a[n] + 1) % 300
        tau, com = oracle.accept_greedy(lg, draft)
        assert tau == n + 1
        assert list(com[:tau]) == list(a[:tau]) and all(c == -1 for c in com[tau:])
        assert list(com[:n]) == list(draft[:n])


def test_planted_geometric_accept_lengths_have_closed_form_mean():
    # min(G-1, 15) with G ~ Geometric(0.3): E[tau] = sum_{i=0}^{15} 0.7^i
    n = inputs.geometric_accept_lengths(200000, 0.3, 15, seed=14).double()
    mean_tau = 1.0 + n.mean().item()
    closed = (1 - 0.7 ** 16) / 0.3
    assert abs(mean_tau - closed) < 4 * (n.std().item() / math.sqrt(200000))
    assert abs((n == 0).double().mean().item() - 0.3) < 0.005


def test_near_tie_gap_helper():
    lg = np.array([[5.0, 4.0, 4.0005, 1.0]], dtype=np.float32)
    assert topk_gap(lg, 1)[0] == pytest.approx(5.0 - 4.0005, rel=1e-6)
    assert topk_gap(lg, 2)[0] == pytest.approx(0.0005, rel=1e-3)
