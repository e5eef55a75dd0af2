"""Python binding of libdfv.so (ctypes).  Argument marshalling only: every step
of the block-verify path runs in the library's CUDA kernels.  Tensors must be
CUDA tensors; calls enqueue work on torch's current CUDA stream."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from .inputs import LayerWeights

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdfv.so")

F32, BF16, MXFP4, Q8, F16 = 0, 1, 2, 3, 4
# device error bits (DFV_DEVERR_* in include/dfv.h)
DEVERR_STAGE_WAIT, DEVERR_SLOT_WAIT, DEVERR_DRAIN_WAIT, DEVERR_GRID_WAIT = 0x1, 0x2, 0x4, 0x8
DEVERR_SCALE_RANGE, DEVERR_REDUCE_WAIT, DEVERR_ROUTING = 0x10, 0x20, 0x40
_NAMES = {"f32": F32, "bf16": BF16, "mxfp4": MXFP4, "q8": Q8}
EXPORTS = ("dfv_version", "dfv_status_string", "dfv_last_error_detail", "dfv_profile_set_events",
           "dfv_read_device_error", "dfv_set_path", "dfv_last_layer_path", "dfv_fused_unavailable_reason",
           "dfv_accept_greedy_noalloc", "dfv_set_staging", "dfv_last_staging",
           "dfv_moe_workspace_size",
           "dfv_route_topk", "dfv_moe_block_forward", "dfv_moe_block_forward_host", "dfv_moe_stack_forward",
           "dfv_accept_workspace_size", "dfv_accept_greedy", "dfv_selftest_bounded_waits", "dfv_selftest_mma",
           "dfv_selftest_tcgen05", "dfv_moe_batch_workspace_size", "dfv_moe_batch_forward",
           "dfv_set_stack_launch")


class DfvError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _load()
        super().__init__("%s: %s: %s" % (where, lib.dfv_status_string(status).decode(),
                                         lib.dfv_last_error_detail().decode()))
        self.status = status


class CLayer(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
        ("d_ff", ctypes.c_int), ("norm_topk", ctypes.c_int),
        ("w_dtype", ctypes.c_int), ("r_dtype", ctypes.c_int),
        ("w_router", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("w_down", ctypes.c_void_p), ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p),
        ("s_down", ctypes.c_void_p), ("n_shared", ctypes.c_int),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libdfv.so is not built (%s); run speculative_decoding_moe_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.dfv_version.restype = I
        L.dfv_status_string.restype = ctypes.c_char_p
        L.dfv_status_string.argtypes = [I]
        L.dfv_last_error_detail.restype = ctypes.c_char_p
        L.dfv_moe_workspace_size.restype = S
        L.dfv_moe_workspace_size.argtypes = [P, I]
        L.dfv_route_topk.argtypes = [P, P, I, I, P, P, P, P, P, P, P, S, P]
        L.dfv_moe_block_forward.argtypes = [P, P, I, I, P, P, P, P, S, P]
        L.dfv_moe_block_forward_host.argtypes = [P, P, I, I, P, P, S, P]
        L.dfv_moe_stack_forward.argtypes = [P, I, P, I, ctypes.c_float, P, P, S, P]
        L.dfv_accept_workspace_size.restype = S
        L.dfv_accept_workspace_size.argtypes = [I, I]
        L.dfv_accept_greedy.argtypes = [P, I, I, I, P, P, P, P, S, P]
        L.dfv_profile_set_events.argtypes = [P, I]
        L.dfv_accept_greedy_noalloc.argtypes = [P, I, I, I, P, P, P, P]
        L.dfv_read_device_error.argtypes = [P, P, P]
        L.dfv_selftest_bounded_waits.argtypes = [P, S, P]
        L.dfv_selftest_mma.argtypes = [I, P, P, P, P]
        L.dfv_selftest_tcgen05.argtypes = [P, P, I, I, P, P, P]
        L.dfv_moe_batch_workspace_size.restype = S
        L.dfv_moe_batch_workspace_size.argtypes = [P, I]
        L.dfv_moe_batch_forward.argtypes = [P, P, I, I, P, P, P, P, S, P]
        L.dfv_set_path.argtypes = [I]
        L.dfv_set_stack_launch.argtypes = [I]
        L.dfv_set_staging.restype = I
        L.dfv_set_staging.argtypes = [I]
        L.dfv_last_staging.restype = I
        L.dfv_last_staging.argtypes = []
        L.dfv_last_layer_path.restype = I
        L.dfv_fused_unavailable_reason.restype = ctypes.c_char_p
        _lib = L
    return _lib


def lib():
    return _load()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _act(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("activations must be bf16 or fp32, got %s" % t.dtype)


def _check(status: int, where: str):
    if status != 0:
        raise DfvError(status, where)


class Layer:
    """A layer descriptor over device-resident weights (keeps them alive)."""

    def __init__(self, w: LayerWeights):
        for t in (w.w_router, w.w_gate, w.w_up, w.w_down):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("layer weights must be contiguous CUDA tensors")
        s = w.shape
        if w.w_gate.shape[0] != s.n_experts + s.n_shared:
            raise ValueError("expert matrices hold %d experts, the shape needs %d routed + %d shared"
                             % (w.w_gate.shape[0], s.n_experts, s.n_shared))
        self.w = w
        self.shape = s
        self.c = CLayer(s.d, s.n_experts, s.top_k, s.d_ff, s.norm_topk, _NAMES[s.w_dtype], _NAMES[s.r_dtype],
                        w.w_router.data_ptr(), w.w_gate.data_ptr(), w.w_up.data_ptr(), w.w_down.data_ptr(),
                        None if w.s_gate is None else w.s_gate.data_ptr(),
                        None if w.s_up is None else w.s_up.data_ptr(),
                        None if w.s_down is None else w.s_down.data_ptr(), s.n_shared)

    @property
    def ref(self):
        return ctypes.byref(self.c)


def workspace_size(layer: Layer, k_max: int) -> int:
    return int(_load().dfv_moe_workspace_size(layer.ref, int(k_max)))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (the library requires zeros before first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def route_topk(layer: Layer, hidden: torch.Tensor, ws: torch.Tensor, stream=None):
    k = hidden.shape[0]
    s = layer.shape
    dev = hidden.device
    idx = torch.empty(k, s.top_k, dtype=torch.int32, device=dev)
    w = torch.empty(k, s.top_k, dtype=torch.float32, device=dev)
    woken = torch.empty(min(s.n_experts, k * s.top_k), dtype=torch.int32, device=dev)
    nw = torch.empty(1, dtype=torch.int32, device=dev)
    offs = torch.empty(min(s.n_experts, k * s.top_k) + 1, dtype=torch.int32, device=dev)
    gat = torch.empty(k * s.top_k, dtype=torch.int32, device=dev)
    st = _load().dfv_route_topk(layer.ref, _p(hidden), _act(hidden), k, _p(idx), _p(w), _p(woken), _p(nw), _p(offs),
                                _p(gat), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dfv_route_topk")
    return dict(topk_idx=idx, topk_w=w, woken=woken, n_woken=nw, offsets=offs, gather=gat)


def moe_block_forward(layer: Layer, hidden: torch.Tensor, ws: torch.Tensor, out: Optional[torch.Tensor] = None,
                      topk_idx: Optional[torch.Tensor] = None, n_woken: Optional[torch.Tensor] = None, stream=None):
    k = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    st = _load().dfv_moe_block_forward(layer.ref, _p(hidden), _act(hidden), k, _p(out), _p(topk_idx), _p(n_woken),
                                       _p(ws), ws.numel(), _stream(stream))
    _check(st, "dfv_moe_block_forward")
    return out


def batch_workspace_size(layer: Layer, n_rows_max: int) -> int:
    return int(_load().dfv_moe_batch_workspace_size(layer.ref, int(n_rows_max)))


def moe_batch_forward(layer: Layer, hidden: torch.Tensor, n_blocks: int, ws: torch.Tensor,
                      out: Optional[torch.Tensor] = None, topk_idx: Optional[torch.Tensor] = None,
                      n_woken: Optional[torch.Tensor] = None, stream=None):
    """n_blocks verify blocks of k = rows / n_blocks positions through one layer."""
    T = hidden.shape[0]
    if T % n_blocks:
        raise ValueError("rows %d are not n_blocks=%d blocks of equal size" % (T, n_blocks))
    if out is None:
        out = torch.empty_like(hidden)
    st = _load().dfv_moe_batch_forward(layer.ref, _p(hidden), n_blocks, T // n_blocks, _p(out), _p(topk_idx),
                                       _p(n_woken), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dfv_moe_batch_forward")
    return out


def moe_block_forward_host(layer: Layer, hidden_host: torch.Tensor, out_host: torch.Tensor, ws: torch.Tensor,
                           stream=None):
    """hidden_host / out_host: CPU tensors (pinned for asynchronous copies)."""
    k = hidden_host.shape[0]
    st = _load().dfv_moe_block_forward_host(layer.ref, _p(hidden_host), _act(hidden_host), k, _p(out_host), _p(ws),
                                            ws.numel(), _stream(stream))
    _check(st, "dfv_moe_block_forward_host")
    return out_host


def moe_stack_forward(layers: Sequence[Layer], x: torch.Tensor, ws: torch.Tensor, eps: float = 1e-6, stream=None,
                      n_woken: Optional[torch.Tensor] = None):
    """x <- the stack applied to x (in place).  n_woken: optional int32 [len(layers)]
    device tensor that receives each layer's routed woken-expert count."""
    arr = (CLayer * len(layers))(*[L.c for L in layers])
    if n_woken is not None and (n_woken.dtype != torch.int32 or n_woken.numel() < len(layers)):
        raise ValueError("n_woken must be int32 with one entry per layer")
    st = _load().dfv_moe_stack_forward(arr, len(layers), _p(x), x.shape[0], float(eps), _p(n_woken), _p(ws),
                                       ws.numel(), _stream(stream))
    _check(st, "dfv_moe_stack_forward")
    return x


def accept_workspace_size(k_max: int, V: int) -> int:
    return int(_load().dfv_accept_workspace_size(int(k_max), int(V)))


def accept_greedy(logits: torch.Tensor, draft: torch.Tensor, ws: torch.Tensor, tau: Optional[torch.Tensor] = None,
                  committed: Optional[torch.Tensor] = None, stream=None):
    rows, V = logits.shape
    k = rows - 1
    dev = logits.device
    if tau is None:
        tau = torch.empty(1, dtype=torch.int32, device=dev)
    if committed is None:
        committed = torch.empty(k + 1, dtype=torch.int32, device=dev)
    st = _load().dfv_accept_greedy(_p(logits), _act(logits), k, V, _p(draft), _p(tau), _p(committed), _p(ws),
                                   ws.numel(), _stream(stream))
    _check(st, "dfv_accept_greedy")
    return tau, committed


def profile_set_events(events: Optional[Sequence[torch.cuda.Event]]):
    """Record the 4 phase-boundary events in later layer calls (None: off)."""
    if events is None:
        _check(_load().dfv_profile_set_events(None, 0), "dfv_profile_set_events")
        return
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(_load().dfv_profile_set_events(arr, len(events)), "dfv_profile_set_events")


def read_device_error(ws: torch.Tensor, stream=None) -> int:
    """Device error bits of a workspace (synchronises the stream)."""
    out = ctypes.c_uint32(0)
    _check(_load().dfv_read_device_error(_p(ws), ctypes.byref(out), _stream(stream)), "dfv_read_device_error")
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return int(out.value)


def selftest_bounded_waits(ws: torch.Tensor, stream=None):
    """Run the bounded-wait self-test on `ws` (about 4 s on the GPU; read the
    error word with read_device_error, then zero-fill ws)."""
    _check(_load().dfv_selftest_bounded_waits(_p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dfv_selftest_bounded_waits")


def selftest_mma(a: torch.Tensor, b: torch.Tensor, stream=None) -> torch.Tensor:
    """D = A . B (16 x 16 x 16) through the expert kernels' MMA fragment path;
    a and b are bf16 or fp16 CUDA tensors [16, 16]."""
    if a.shape != (16, 16) or b.shape != (16, 16) or a.dtype != b.dtype:
        raise ValueError("A and B must be [16, 16] tensors of one dtype")
    code = {torch.bfloat16: BF16, torch.float16: F16}.get(a.dtype)
    if code is None:
        raise TypeError("A and B must be bf16 or fp16, got %s" % a.dtype)
    a, b = a.contiguous(), b.contiguous()
    out = torch.empty(16, 16, dtype=torch.float32, device=a.device)
    _check(_load().dfv_selftest_mma(code, _p(a), _p(b), _p(out), _stream(stream)), "dfv_selftest_mma")
    return out


def selftest_tcgen05(a: torch.Tensor, b: torch.Tensor, stream=None):
    """D = A . B^T (A [128, K], B [N, K], bf16) through the tcgen05 / TMEM path;
    returns (D [128, N] fp32, status)."""
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16 or a.shape[0] != 128 or a.shape[1] != b.shape[1]:
        raise ValueError("A must be [128, K] and B [N, K], both bf16")
    a, b = a.contiguous(), b.contiguous()
    d = torch.full((128, b.shape[0]), float("nan"), dtype=torch.float32, device=a.device)
    st = torch.zeros(1, dtype=torch.int32, device=a.device)
    _check(_load().dfv_selftest_tcgen05(_p(a), _p(b), b.shape[0], a.shape[1], _p(d), _p(st), _stream(stream)),
           "dfv_selftest_tcgen05")
    return d, st


def set_staging(max_mode: int):
    """Highest gate/up staging mode of the single-launch bf16 kernel (3, the default, 2, 1 or 0)."""
    _check(_load().dfv_set_staging(int(max_mode)), "dfv_set_staging")


def last_staging() -> int:
    return int(_load().dfv_last_staging())


def set_path(fused: bool):
    """Select the fused single-launch layer kernel (default) or the multi-kernel path."""
    _check(_load().dfv_set_path(1 if fused else 0), "dfv_set_path")


def set_stack_launch(mode):
    """Stacks whose layers allow it: 0 (or False) one launch per layer; 1 (default) one persistent
    launch per 48 layers for eager calls with k <= 8 (per layer inside a CUDA graph); 2 (or True)
    one persistent launch per 48 layers for every k."""
    m = {False: 0, True: 2}.get(mode, mode) if isinstance(mode, bool) else int(mode)
    _check(_load().dfv_set_stack_launch(m), "dfv_set_stack_launch")


def last_layer_path() -> int:
    """Path of the last layer call from this thread: 1 fused, 0 multi-kernel, 2 batched, 3 persistent stack."""
    return int(_load().dfv_last_layer_path())


def fused_unavailable_reason() -> str:
    return _load().dfv_fused_unavailable_reason().decode()


def accept_greedy_noalloc(logits: torch.Tensor, draft: torch.Tensor, tau: Optional[torch.Tensor] = None,
                          committed: Optional[torch.Tensor] = None, stream=None):
    """Greedy acceptance with the library's fixed device scratch (no workspace)."""
    rows, V = logits.shape
    k = rows - 1
    dev = logits.device
    if tau is None:
        tau = torch.empty(1, dtype=torch.int32, device=dev)
    if committed is None:
        committed = torch.empty(k + 1, dtype=torch.int32, device=dev)
    st = _load().dfv_accept_greedy_noalloc(_p(logits), _act(logits), k, V, _p(draft), _p(tau), _p(committed),
                                           _stream(stream))
    _check(st, "dfv_accept_greedy_noalloc")
    return tau, committed
