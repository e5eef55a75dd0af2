"""Helpers shared by the tests: tensor <-> numpy marshalling for the oracle and
near-tie rejection of synthetic router inputs (decided with the oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_moe_gb300 import inputs

_CODE = {"f32": oracle.F32, "bf16": oracle.BF16, "mxfp4": oracle.MXFP4, "q8": oracle.Q8}


def np_of(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view of a tensor; bf16 becomes its uint16 bit patterns."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_layer(lw: inputs.LayerWeights) -> oracle.Layer:
    s = lw.shape
    return oracle.Layer(
        d=s.d, n_experts=s.n_experts, top_k=s.top_k, d_ff=s.d_ff,
        w_dtype=_CODE[s.w_dtype], r_dtype=_CODE[s.r_dtype],
        w_router=np_of(lw.w_router), w_gate=np_of(lw.w_gate), w_up=np_of(lw.w_up), w_down=np_of(lw.w_down),
        s_gate=None if lw.s_gate is None else np_of(lw.s_gate),
        s_up=None if lw.s_up is None else np_of(lw.s_up),
        s_down=None if lw.s_down is None else np_of(lw.s_down),
        norm_topk=s.norm_topk, n_shared=s.n_shared)


def topk_gap(logits: np.ndarray, K: int) -> np.ndarray:
    """Per row: (K-th largest logit) - ((K+1)-th largest logit)."""
    srt = -np.sort(-logits.astype(np.float64), axis=1)
    if K >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    return srt[:, K - 1] - srt[:, K]


def hidden_without_near_ties(ol: oracle.Layer, k: int, act: str, seed: int, mode: str = "independent",
                             min_gap: float = 1e-3, device="cpu", max_attempts: int = 200) -> torch.Tensor:
    """Draw hidden[k, d]; redraw (seed, attempt) until every row's gap between
    the K-th and (K+1)-th router logit (oracle, fp32) is at least min_gap."""
    for attempt in range(max_attempts):
        x = inputs.make_hidden(k, ol.d, act, seed * 1000 + attempt, mode=mode, device=device)
        logits, _, _ = oracle.route(ol, np_of(x))
        if np.all(topk_gap(logits, ol.top_k) >= min_gap):
            return x
    raise RuntimeError("no near-tie-free draw in %d attempts" % max_attempts)
