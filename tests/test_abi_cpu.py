"""The C-ABI library builds, loads and exports every symbol include/dfv.h
declares; host-side argument validation rejects bad calls before any CUDA
call (so these run without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_moe_gb300 import build as b
    b.build()
    from speculative_decoding_moe_gb300 import dfv
    return dfv


def _declared():
    src = open(os.path.join(ROOT, "include", "dfv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dfv_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    L = lib.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(lib.EXPORTS)


def test_status_strings_and_version(lib):
    L = lib.lib()
    assert L.dfv_version() == 2
    assert L.dfv_status_string(0) == b"DFV_OK"
    assert L.dfv_status_string(3) == b"DFV_ERR_WORKSPACE"


def _layer(lib, **kw):
    c = dict(d=2048, n_experts=128, top_k=8, d_ff=768, norm_topk=1, w_dtype=1, r_dtype=1,
             w_router=0x10000, w_gate=0x20000, w_up=0x30000, w_down=0x40000)
    c.update(kw)
    sc = c.get("scales", (None, None, None))
    return lib.CLayer(c["d"], c["n_experts"], c["top_k"], c["d_ff"], c["norm_topk"], c["w_dtype"], c["r_dtype"],
                      c["w_router"], c["w_gate"], c["w_up"], c["w_down"], *sc, c.get("n_shared", 0))


def test_workspace_sizes(lib):
    L = lib.lib()
    ly = _layer(lib)
    s16 = L.dfv_moe_workspace_size(ctypes.byref(ly), 16)
    s1 = L.dfv_moe_workspace_size(ctypes.byref(ly), 1)
    assert 0 < s1 < s16 < 8 << 20
    assert L.dfv_moe_workspace_size(ctypes.byref(ly), 0) == 0
    assert L.dfv_moe_workspace_size(ctypes.byref(ly), 17) == 0
    assert L.dfv_accept_workspace_size(16, 151936) > 0
    assert L.dfv_accept_workspace_size(17, 151936) == 0
    # a shared expert adds one pair slot per row: K+1 rows of h and ys per token
    sh = L.dfv_moe_workspace_size(ctypes.byref(_layer(lib, n_shared=1)), 16)
    assert sh - s16 >= 16 * (2048 + 768) * 4
    assert L.dfv_moe_workspace_size(ctypes.byref(_layer(lib, n_shared=2)), 16) == 0
    assert L.dfv_moe_workspace_size(ctypes.byref(_layer(lib, n_shared=-1)), 16) == 0


@pytest.mark.parametrize("kw,k,status", [
    (dict(), 0, 1),                      # k out of range
    (dict(), 17, 1),
    (dict(top_k=9), 4, 2),               # K > 8
    (dict(n_experts=4, top_k=5), 4, 2),  # K > E
    (dict(n_experts=257), 4, 2),
    (dict(d=2000), 4, 2),                # d % 32
    (dict(w_dtype=0), 4, 2),             # f32 experts with bf16 activations
    (dict(w_router=0x10001), 4, 1),      # misaligned weight
    (dict(w_gate=0), 4, 1),              # NULL weight
    (dict(w_dtype=2), 4, 1),             # mxfp4 experts without scales
    (dict(w_dtype=2, d=2080, scales=(0x81000, 0x82000, 0x83000)), 4, 2),   # mxfp4 needs d % 64
    (dict(w_dtype=2, d_ff=736, scales=(0x81000, 0x82000, 0x83000)), 4, 2),  # and d_ff % 64
    (dict(w_dtype=2, r_dtype=0, scales=(0x81000, 0x82000, 0x83000)), 4, 2),  # fp32 router with mxfp4
    (dict(n_shared=2), 4, 2),            # at most one shared expert
    (dict(n_shared=-1), 4, 1),
])
def test_invalid_arguments_are_rejected_before_launch(lib, kw, k, status):
    L = lib.lib()
    ly = _layer(lib, **kw)
    st = L.dfv_moe_block_forward(ctypes.byref(ly), ctypes.c_void_p(0x50000), 1, k, ctypes.c_void_p(0x60000), None,
                                 None, ctypes.c_void_p(0x70000), 1 << 30, None)
    assert st == status, L.dfv_last_error_detail()
    assert L.dfv_last_error_detail()


def test_workspace_checks(lib):
    L = lib.lib()
    ly = _layer(lib)
    st = L.dfv_moe_block_forward(ctypes.byref(ly), ctypes.c_void_p(0x50000), 1, 4, ctypes.c_void_p(0x60000), None,
                                 None, ctypes.c_void_p(0x70000), 1024, None)
    assert st == 3
    st = L.dfv_moe_block_forward(ctypes.byref(ly), ctypes.c_void_p(0x50000), 1, 4, ctypes.c_void_p(0x60000), None,
                                 None, ctypes.c_void_p(0x70010), 1 << 30, None)
    assert st == 3
    st = L.dfv_accept_greedy(ctypes.c_void_p(0x50000), 1, 4, 100, ctypes.c_void_p(0x60000),
                             ctypes.c_void_p(0x70000), None, ctypes.c_void_p(0x80000), 8, None)
    assert st == 3
    st = L.dfv_accept_greedy(ctypes.c_void_p(0x50000), 2, 4, 100, ctypes.c_void_p(0x60000),
                             ctypes.c_void_p(0x70000), None, ctypes.c_void_p(0x80000), 1 << 20, None)
    assert st == 2


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_moe_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt and "orc_" not in txt, f


def test_device_error_bits_match_the_header(lib):
    src = open(os.path.join(ROOT, "include", "dfv.h")).read()
    bits = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define DFV_DEVERR_([A-Z_]+) (0x[0-9a-fA-F]+)u", src)}
    assert bits == {"STAGE_WAIT": 1, "SLOT_WAIT": 2, "DRAIN_WAIT": 4, "GRID_WAIT": 8, "SCALE_RANGE": 16,
                    "REDUCE_WAIT": 32, "ROUTING": 64}
    for name, v in bits.items():
        assert getattr(lib, "DEVERR_" + name) == v


def test_staging_mode_is_validated(lib):
    L = lib.lib()
    assert L.dfv_set_staging(4) == 1
    assert L.dfv_set_staging(-1) == 1
    assert L.dfv_set_staging(2) == 0
    assert L.dfv_set_staging(3) == 0  # the default again
    assert L.dfv_last_staging() == -1


def test_selftest_entry_point_validates_its_workspace(lib):
    L = lib.lib()
    assert L.dfv_selftest_bounded_waits(None, 1 << 20, None) == 3
    assert L.dfv_selftest_bounded_waits(ctypes.c_void_p(0x70010), 1 << 20, None) == 3  # not 256-aligned
    assert L.dfv_selftest_bounded_waits(ctypes.c_void_p(0x70000), 4096, None) == 3      # under the 8 KB of counters
    assert L.dfv_last_error_detail()
