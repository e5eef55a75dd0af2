"""Planted mistakes in the CPU oracle, for showing that a pin catches them.

A mutant is oracle/oracle.c with one exact source fragment replaced, compiled
with gcc into a temporary directory and loaded with ctypes.  Nothing here is
used by the oracle itself or by the CUDA library; the tests only compare a
mutant's output with the closed form a pin states."""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

import oracle

_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def build_mutant(old: str, new: str):
    """Compile oracle.c with the single occurrence of `old` replaced by `new`."""
    with open(os.path.join(_SRC, "oracle.c")) as f:
        text = f.read()
    assert text.count(old) == 1, "the fragment to mutate must occur exactly once: %r" % old
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    src = os.path.join(tmp, "oracle.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    so = os.path.join(tmp, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off", "-I", _SRC, src, "-o", so,
                    "-lm"], check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.orc_moe_forward.argtypes = [P, P, I, I, P, I]
    return lib


def moe_forward_with(lib, layer: oracle.Layer, x: np.ndarray) -> np.ndarray:
    """orc_moe_forward of a (possibly mutated) oracle library."""
    k = x.shape[0]
    out = np.empty((k, layer.d), dtype=np.float64)
    lc = layer.c()
    code = oracle.F32 if x.dtype == np.float32 else oracle.BF16
    rc = lib.orc_moe_forward(ctypes.byref(lc), x.ctypes.data_as(ctypes.c_void_p), code, k,
                             out.ctypes.data_as(ctypes.c_void_p), 1)
    if rc:
        raise ValueError("orc_moe_forward failed (%d)" % rc)
    return out


def matmul_with(lib, dtype: int, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """orc_matmul of a (possibly mutated) oracle library (operands as in oracle.matmul)."""
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.orc_matmul.argtypes = [I, P, P, I, I, I, P]
    M, L = a.shape
    N = b.shape[1]
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    out = np.empty((M, N), dtype=np.float64)
    rc = lib.orc_matmul(int(dtype), a.ctypes.data_as(P), b.ctypes.data_as(P), M, L, N, out.ctypes.data_as(P))
    if rc:
        raise ValueError("orc_matmul failed (%d)" % rc)
    return out
