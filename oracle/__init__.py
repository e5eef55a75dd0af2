"""Plain CPU oracle for the MoE block-verify step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
``libdfv.so`` and its Python binding) never imports, links or calls it, and the
two share no code.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double precision, loops in
the order the definitions state them).  This module only compiles that file
with gcc and marshals numpy arrays across ctypes.

Sources, by page title and section:
  * "Speculating on a Strix Halo", sections "Speculative decoding" (greedy
    acceptance, committed length), "What the pieces cost" (per-token routing,
    woken-expert union, the always-on shared expert), "The verify's own cost"
    (tokens sorted by expert), reference 1 (256 experts, 8 routed plus 1
    shared activated).
  * "Speculating on a Strix Halo (part 2)", sections "The verification cog"
    and "Why drafter performance doesn't really matter" (prefix acceptance).
  * the MI355X / vLLM DFlash write-up (allbreaknews.com/?p=4397), sections
    "Why Quantize the Target Model on Top?" and "Results: Quantizing the Target
    Model" (mxfp4 target weights).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

F32, BF16, MXFP4, Q8, F16 = 0, 1, 2, 3, 4
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP when available)."""
    src = os.path.join(_HERE, "oracle.c")
    hdr = os.path.join(_HERE, "oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
        ("d_ff", ctypes.c_int), ("norm_topk", ctypes.c_int),
        ("w_dtype", ctypes.c_int), ("r_dtype", ctypes.c_int),
        ("w_router", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("w_down", ctypes.c_void_p), ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p),
        ("s_down", ctypes.c_void_p), ("n_shared", ctypes.c_int),
    ]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_bf16_to_double.restype = D
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_double_to_bf16.restype = ctypes.c_uint16
        L.orc_double_to_bf16.argtypes = [D]
        L.orc_e2m1_value.restype = D
        L.orc_e2m1_value.argtypes = [I]
        L.orc_e8m0_value.restype = D
        L.orc_e8m0_value.argtypes = [I]
        L.orc_fp16_to_double.restype = D
        L.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_silu.restype = D
        L.orc_silu.argtypes = [D]
        L.orc_decode_rows.argtypes = [I, P, P, I, I, I, P]
        L.orc_route.argtypes = [P, P, I, I, P, P, P]
        L.orc_matmul.argtypes = [I, P, P, I, I, I, P]
        L.orc_woken.argtypes = [I, I, I, P, P, P, P, P]
        L.orc_expert_ffn.argtypes = [P, I, P, P]
        L.orc_moe_forward.argtypes = [P, P, I, I, P, I]
        L.orc_rmsnorm.argtypes = [P, I, I, I, D, P]
        L.orc_stack_forward.argtypes = [P, I, P, I, D, P, I]
        L.orc_argmax_rows.argtypes = [P, I, I, I, P]
        L.orc_accept_greedy.argtypes = [P, I, I, I, P, P, P]
        L.orc_num_threads_available.restype = I
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("activations must be float32 or uint16 (bf16 bit patterns), got %s" % a.dtype)


@dataclass
class Layer:
    """One MoE layer's weights as numpy arrays.

    bf16 arrays hold raw uint16 bit patterns; mxfp4 matrices hold packed
    nibbles (uint8, low nibble = even column) plus e8m0 scales (uint8, one per
    32 consecutive elements of a row); q8 matrices hold int8 codes plus one
    float16 scale per 32 consecutive elements of a row.
    """
    d: int
    n_experts: int
    top_k: int
    d_ff: int
    w_dtype: int
    r_dtype: int
    w_router: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray
    s_gate: Optional[np.ndarray] = None
    s_up: Optional[np.ndarray] = None
    s_down: Optional[np.ndarray] = None
    norm_topk: int = 1
    n_shared: int = 0   # 1: one always-on shared expert, stored as expert n_experts

    def c(self) -> _Layer:
        arrs = [self.w_router, self.w_gate, self.w_up, self.w_down, self.s_gate, self.s_up, self.s_down]
        for a in arrs:
            if a is not None:
                assert a.flags["C_CONTIGUOUS"]
        return _Layer(self.d, self.n_experts, self.top_k, self.d_ff, self.norm_topk,
                      self.w_dtype, self.r_dtype, *[(_ptr(a).value if a is not None else None) for a in arrs],
                      self.n_shared)


# ---------------------------------------------------------------- scalars
def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(int(bits))


def double_to_bf16(v: float) -> int:
    return int(lib().orc_double_to_bf16(float(v)))


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e8m0_value(e: int) -> float:
    return lib().orc_e8m0_value(int(e))


def fp16_to_double(bits: int) -> float:
    return lib().orc_fp16_to_double(int(bits))


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def decode_rows(dtype: int, data: np.ndarray, scales: Optional[np.ndarray], r0: int, nrows: int, cols: int) -> np.ndarray:
    out = np.empty((nrows, cols), dtype=np.float64)
    rc = lib().orc_decode_rows(dtype, _ptr(data), _ptr(scales), r0, nrows, cols, _ptr(out))
    if rc:
        raise ValueError("orc_decode_rows failed (%d)" % rc)
    return out


def matmul(dtype: int, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """D = A . B in double from operands of one element format (F32 as
    float32, BF16 / F16 as their uint16 bit patterns)."""
    M, L = a.shape
    L2, N = b.shape
    assert L == L2
    out = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_matmul(int(dtype), _ptr(np.ascontiguousarray(a)), _ptr(np.ascontiguousarray(b)), M, L, N, _ptr(out))
    if rc:
        raise ValueError("orc_matmul failed (%d)" % rc)
    return out


# ---------------------------------------------------------------- routing
def route(layer: Layer, x: np.ndarray):
    """-> (logits[k,E] float32, topk_idx[k,K] int32, topk_w[k,K] float64)"""
    k = x.shape[0]
    lc = layer.c()
    logits = np.empty((k, layer.n_experts), dtype=np.float32)
    idx = np.empty((k, layer.top_k), dtype=np.int32)
    w = np.empty((k, layer.top_k), dtype=np.float64)
    rc = lib().orc_route(ctypes.byref(lc), _ptr(x), _dtype_code(x), k, _ptr(logits), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("orc_route failed (%d)" % rc)
    return logits, idx, w


def woken(topk_idx: np.ndarray, n_experts: int):
    """-> (woken[W], offsets[W+1], gather[k*K]) as int32 arrays"""
    k, K = topk_idx.shape
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    wk = np.empty(n_experts, dtype=np.int32)
    nw = np.zeros(1, dtype=np.int32)
    offs = np.empty(n_experts + 1, dtype=np.int32)
    gat = np.empty(k * K, dtype=np.int32)
    rc = lib().orc_woken(k, K, n_experts, _ptr(idx), _ptr(wk), _ptr(nw), _ptr(offs), _ptr(gat))
    if rc < 0:
        raise ValueError("orc_woken failed (%d)" % rc)
    W = int(nw[0])
    return wk[:W].copy(), offs[:W + 1].copy(), gat


def expert_ffn(layer: Layer, e: int, x_row: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_row, dtype=np.float64)
    y = np.empty(layer.d, dtype=np.float64)
    lc = layer.c()
    rc = lib().orc_expert_ffn(ctypes.byref(lc), int(e), _ptr(x), _ptr(y))
    if rc:
        raise ValueError("orc_expert_ffn failed (%d)" % rc)
    return y


def moe_forward(layer: Layer, x: np.ndarray, nthreads: int = 1) -> np.ndarray:
    """MoE output of one layer (routed experts + the shared expert when
    layer.n_shared), float64 [k, d]."""
    k = x.shape[0]
    out = np.empty((k, layer.d), dtype=np.float64)
    lc = layer.c()
    rc = lib().orc_moe_forward(ctypes.byref(lc), _ptr(x), _dtype_code(x), k, _ptr(out), int(nthreads))
    if rc:
        raise ValueError("orc_moe_forward failed (%d)" % rc)
    return out


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    k, d = x.shape
    out = np.empty((k, d), dtype=np.float64)
    rc = lib().orc_rmsnorm(_ptr(x), _dtype_code(x), k, d, float(eps), _ptr(out))
    if rc:
        raise ValueError("orc_rmsnorm failed (%d)" % rc)
    return out


def stack_forward(layers, x: np.ndarray, eps: float = 1e-6, nthreads: int = 1) -> np.ndarray:
    """Pre-norm residual stack over bf16 residual stream x[k,d] (uint16) -> uint16."""
    assert x.dtype == np.uint16
    k = x.shape[0]
    cl = (_Layer * len(layers))(*[L.c() for L in layers])
    out = np.empty_like(x)
    rc = lib().orc_stack_forward(cl, len(layers), _ptr(x), k, float(eps), _ptr(out), int(nthreads))
    if rc:
        raise ValueError("orc_stack_forward failed (%d)" % rc)
    return out


# ---------------------------------------------------------------- acceptance
def argmax_rows(logits: np.ndarray) -> np.ndarray:
    rows, V = logits.shape
    a = np.empty(rows, dtype=np.int32)
    rc = lib().orc_argmax_rows(_ptr(logits), _dtype_code(logits), rows, V, _ptr(a))
    if rc:
        raise ValueError("orc_argmax_rows failed (%d)" % rc)
    return a


def accept_greedy(logits: np.ndarray, draft: np.ndarray):
    """-> (tau, committed[k+1]) with committed[i] = -1 past the bonus token."""
    rows, V = logits.shape
    k = rows - 1
    dr = np.ascontiguousarray(draft, dtype=np.int32)
    assert dr.shape == (k,)
    tau = np.zeros(1, dtype=np.int32)
    com = np.empty(k + 1, dtype=np.int32)
    rc = lib().orc_accept_greedy(_ptr(logits), _dtype_code(logits), k, V, _ptr(dr), _ptr(tau), _ptr(com))
    if rc:
        raise ValueError("orc_accept_greedy failed (%d)" % rc)
    return int(tau[0]), com


def num_threads_available() -> int:
    return int(lib().orc_num_threads_available())
