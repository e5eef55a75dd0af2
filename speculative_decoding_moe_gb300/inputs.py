"""Seeded synthetic inputs for the MoE block-verify workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no routing, no expert FFN, no argmax).  Both the CUDA
path's tests/bench and the CPU oracle's tests take their inputs from here.

Shapes and distributions follow the workloads the method's write-ups describe
("Speculating on a Strix Halo", section "What the pieces cost": 16-token
blocks, 8 routed experts per token; the MI355X / vLLM write-up: mxfp4 target
weights), scaled to one layer:

* ``tiny``      d=256, E=16, top-2, d_ff=128, fp32 weights ~N(0, 0.02), router
                ~N(0, 0.05), hidden ~N(0, 1), k=4; logits[5, 1024] ~N(0, 1).
* ``a3b``       d=2048, E=128, top-8, d_ff=768, bf16 weights ~N(0, 0.02), router
                ~N(0, 0.02), renormalised top-k weights, k in 1..16.
* ``mxfp4``     d=2048, E=256, top-8, d_ff=512, e2m1 codes uniform over the 16
                nibbles, e8m0 scales uniform in 2^{-8..0}, bf16 router
                ~N(0, 0.02), bf16 activations.
* ``q8``        the mxfp4 layer's shape with 8-bit weights: int8 codes uniform
                over [-127, 127], one binary16 scale per 32 elements uniform in
                w_std/73.3 * [0.5, 1.5) (weights of the other layers' spread).
* ``e256+shared`` d=2048, E=256, top-8, d_ff=512, bf16, plus one always-on
                shared expert of the same size ("What the pieces cost"; the
                model card it cites: 8 routed plus 1 shared activated).
* acceptance    logits[k+1, V] ~N(0, s) with drafts planted so the accepted
                prefix length is Geometric(0.3) - 1, capped at k - 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = ("f32", "bf16", "mxfp4", "q8")


@dataclass(frozen=True)
class LayerShape:
    d: int
    n_experts: int
    top_k: int
    d_ff: int
    w_dtype: str = "bf16"      # expert weights: f32 | bf16 | mxfp4 | q8
    r_dtype: str = "bf16"      # router weights: f32 | bf16
    act: str = "bf16"          # activations:    f32 | bf16
    w_std: float = 0.02
    r_std: float = 0.02
    scale_exp: tuple = (119, 127)   # e8m0 exponent range (inclusive), mxfp4 only
    norm_topk: int = 1
    n_shared: int = 0               # 1: one always-on shared expert (expert index E)


TINY = LayerShape(d=256, n_experts=16, top_k=2, d_ff=128, w_dtype="f32", r_dtype="f32", act="f32",
                  w_std=0.02, r_std=0.05)
A3B = LayerShape(d=2048, n_experts=128, top_k=8, d_ff=768)
MXFP4 = LayerShape(d=2048, n_experts=256, top_k=8, d_ff=512, w_dtype="mxfp4")
# the same layer with 8-bit weights (int8 codes, one binary16 scale per 32 elements)
Q8 = LayerShape(d=2048, n_experts=256, top_k=8, d_ff=512, w_dtype="q8")
# 256 routed experts (top-8) plus one always-on shared expert of the same size
E256_SHARED = LayerShape(d=2048, n_experts=256, top_k=8, d_ff=512, n_shared=1)


def _torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


@dataclass
class LayerWeights:
    """One layer's weights as torch tensors (any device).

    f32/bf16: w_gate, w_up [E', d_ff, d]; w_down [E', d, d_ff].
    mxfp4:    w_gate, w_up uint8 [E', d_ff, d/2]; w_down uint8 [E', d, d_ff/2]
              (low nibble = even column) and s_* uint8 e8m0 scales
              [E', rows, cols/32].
    q8:       w_gate, w_up int8 [E', d_ff, d]; w_down int8 [E', d, d_ff] and
              s_* float16 scales [E', rows, cols/32].
    E' = E + n_shared: the shared expert, if any, is the last one.  The
    router is [E, d].
    """
    shape: LayerShape
    w_router: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    s_gate: Optional[torch.Tensor] = None
    s_up: Optional[torch.Tensor] = None
    s_down: Optional[torch.Tensor] = None

    def to(self, device) -> "LayerWeights":
        f = lambda t: None if t is None else t.to(device)
        return LayerWeights(self.shape, f(self.w_router), f(self.w_gate), f(self.w_up), f(self.w_down),
                            f(self.s_gate), f(self.s_up), f(self.s_down))

    def expert_bytes(self) -> int:
        """HBM bytes of one expert's gate+up+down weights (and scales)."""
        s = self.shape
        per = 0
        for t in (self.w_gate, self.w_up, self.w_down, self.s_gate, self.s_up, self.s_down):
            if t is not None:
                per += t.numel() * t.element_size()
        return per // (s.n_experts + s.n_shared)

    def router_bytes(self) -> int:
        return self.w_router.numel() * self.w_router.element_size()


def make_layer(shape: LayerShape, seed: int, device="cpu") -> LayerWeights:
    g = _gen(seed, device)
    E, d, I = shape.n_experts, shape.d, shape.d_ff
    wr = (torch.randn(E, d, generator=g, device=device) * shape.r_std).to(_torch_dtype(shape.r_dtype))
    E = shape.n_experts + shape.n_shared  # expert matrices: routed experts, then the shared one
    if shape.w_dtype in ("f32", "bf16"):
        dt = _torch_dtype(shape.w_dtype)
        wg = (torch.randn(E, I, d, generator=g, device=device) * shape.w_std).to(dt)
        wu = (torch.randn(E, I, d, generator=g, device=device) * shape.w_std).to(dt)
        wd = (torch.randn(E, d, I, generator=g, device=device) * shape.w_std).to(dt)
        return LayerWeights(shape, wr, wg, wu, wd)
    if shape.w_dtype == "mxfp4":
        assert d % 64 == 0 and I % 64 == 0
        lo, hi = shape.scale_exp
        u8 = torch.uint8

        def codes(rows, cols):
            # two independent uniform nibbles per byte == one uniform byte
            return torch.randint(0, 256, (E, rows, cols // 2), generator=g, device=device, dtype=torch.int32).to(u8)

        def scales(rows, cols):
            return torch.randint(lo, hi + 1, (E, rows, cols // 32), generator=g, device=device, dtype=torch.int32).to(u8)

        wg, sg = codes(I, d), scales(I, d)
        wu, su = codes(I, d), scales(I, d)
        wd, sd = codes(d, I), scales(d, I)
        return LayerWeights(shape, wr, wg, wu, wd, sg, su, sd)
    if shape.w_dtype == "q8":
        assert d % 32 == 0 and I % 32 == 0

        def q8_codes(rows, cols):
            return torch.randint(-127, 128, (E, rows, cols), generator=g, device=device, dtype=torch.int32).to(torch.int8)

        def q8_scales(rows, cols):
            # codes uniform over [-127, 127] spread about 73.3; scales around
            # w_std / 73.3 give weights of about the other layers' spread
            u = torch.rand(E, rows, cols // 32, generator=g, device=device)
            return (shape.w_std / 73.3 * (0.5 + u)).to(torch.float16)

        wg, sg = q8_codes(I, d), q8_scales(I, d)
        wu, su = q8_codes(I, d), q8_scales(I, d)
        wd, sd = q8_codes(d, I), q8_scales(d, I)
        return LayerWeights(shape, wr, wg, wu, wd, sg, su, sd)
    raise ValueError(shape.w_dtype)


def make_hidden(k: int, d: int, act: str, seed: int, mode: str = "independent", device="cpu",
                pert_std: float = 0.3) -> torch.Tensor:
    """hidden[k, d]: independent N(0,1) rows, or a repeated-token block
    (one base vector ~N(0,1) plus per-position N(0, pert_std^2) noise)."""
    g = _gen(seed, device)
    if mode == "independent":
        x = torch.randn(k, d, generator=g, device=device)
    elif mode == "repeated":
        base = torch.randn(1, d, generator=g, device=device)
        x = base + pert_std * torch.randn(k, d, generator=g, device=device)
    else:
        raise ValueError(mode)
    return x.to(_torch_dtype(act))


def make_logits(rows: int, V: int, dtype: str, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(rows, V, generator=g, device=device) * std).to(_torch_dtype(dtype))


def geometric_accept_lengths(n: int, p: float, cap: int, seed: int) -> torch.Tensor:
    """n draws of min(G - 1, cap), G ~ Geometric(p) on {1, 2, ...}."""
    g = _gen(seed, "cpu")
    u = torch.rand(n, generator=g, dtype=torch.float64)
    # inverse CDF of the geometric law on {1, 2, ...}: G = ceil(log(1-u) / log(1-p))
    G = torch.ceil(torch.log1p(-u) / torch.log1p(torch.tensor(-p, dtype=torch.float64))).clamp_min(1)
    return (G.to(torch.int64) - 1).clamp_max(cap).to(torch.int32)


def plant_draft(target_tokens: torch.Tensor, n_accept: int, V: int, seed: int) -> torch.Tensor:
    """draft[k] that agrees with target_tokens[0..n_accept) and differs at
    position n_accept (when n_accept < k); later positions are uniform random.
    ``target_tokens`` (the row-wise argmax of the logits) is supplied by the
    caller."""
    k = target_tokens.numel() - 1
    g = _gen(seed, "cpu")
    draft = torch.randint(0, V, (k,), generator=g, dtype=torch.int32)
    t = target_tokens.to("cpu", torch.int32)
    if n_accept > 0:
        draft[:n_accept] = t[:n_accept]
    if n_accept < k:
        draft[n_accept] = (t[n_accept] + 1) % V
    return draft


def spiked_logits(rows: int, V: int, dtype: str, std: float, seed: int, device="cpu"):
    """Logits ~N(0, std) clamped to [-8 std, 8 std] with one planted entry per
    row set to 9 std, so the row maximum is known by construction.
    Returns (logits, tokens) with tokens[i] the planted column of row i."""
    g = _gen(seed, device)
    x = (torch.randn(rows, V, generator=g, device=device) * std).clamp(-8 * std, 8 * std)
    tok = torch.randint(0, V, (rows,), generator=g, device=device)
    x[torch.arange(rows, device=device), tok] = 9 * std
    return x.to(_torch_dtype(dtype)), tok.to(torch.int32)
