"""The C-ABI library builds, loads and exports every declared symbol (no GPU needed).

Only host-side calls run here: sizes, status strings and argument checks that
return before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from quantized_moe_expert_05_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fm():
    build.build()
    from quantized_moe_expert_05_b300 import fmoe
    return fmoe


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fmoe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(fm):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(fm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/fmoe.h but not exported"


def test_library_is_sm103a_build():
    # the build flags name the B300 architecture only
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.NVCC_FLAGS)


@pytest.mark.parametrize("bits,H,I", [(4, 512, 128), (4, 4096, 1024), (2, 4096, 1024), (4, 2048, 512),
                                      (2, 192, 320), (4, 64, 64)])
def test_expert_bytes_matches_oracle_layout(fm, bits, H, I):
    assert fm.expert_bytes(bits, H, I) == oracle.layout(bits, H, I)[1]


def test_expert_bytes_rejects_bad_shapes(fm):
    assert fm.expert_bytes(3, 512, 128) == 0
    assert fm.expert_bytes(4, 500, 128) == 0
    assert fm.expert_bytes(4, 512, 128, group=32) == 0


def test_status_strings(fm):
    for s in range(6):
        assert fm.status_string(s)
    assert fm.status_string(fm.ERR_TIMEOUT) == "device-side wait timed out"


def test_argument_checks_before_any_launch(fm):
    lib = fm.lib
    L = fm.fmoe_layer()
    L.bits, L.group, L.hidden, L.inter, L.n_experts, L.has_shared = 4, 64, 512, 128, 8, 0
    L.experts = None
    assert lib.fmoe_moe_block(ctypes.byref(L), None, None, None, None, 1, 2, None, None) == fm.ERR_INVALID_ARG
    L.experts = 4096 * 16
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 16, 1, 2, None, None) == fm.ERR_INVALID_ARG
    L.bits = 3
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 32, 1, 2, 256, None) == fm.ERR_UNSUPPORTED
    L.bits, L.group = 4, 32
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 32, 1, 2, 256, None) == fm.ERR_UNSUPPORTED
    L.group = 64
    # K > E, T > 16, misaligned workspace
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 4096, 1, 9, 256, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 4096, 17, 2, 256, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_moe_block(ctypes.byref(L), 16, 16, 16, 4096, 1, 2, 128, None) == fm.ERR_INVALID_ARG
    # out overlapping x
    assert lib.fmoe_moe_block(ctypes.byref(L), 4096, 1 << 20, 1 << 21, 4096 + 512, 1, 2, 256,
                              None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_route(None, 1, 8, 2, 16, 16, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_route(16, 1, 8, 9, 16, 16, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_route(16, 1, 2000, 2, 16, 16, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_stack_decode(None, 1, 16, 16, 2, 1e-6, 256, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_debug_wait_test(256, 0, 1, 10, None) == fm.ERR_INVALID_ARG


def test_workspace_bytes(fm):
    L = fm.fmoe_layer()
    L.bits, L.group, L.hidden, L.inter, L.n_experts, L.has_shared = 4, 64, 4096, 1024, 512, 1
    a = fm.lib.fmoe_workspace_bytes(ctypes.byref(L), 1, 4, 1)
    b = fm.lib.fmoe_workspace_bytes(ctypes.byref(L), 16, 4, 1)
    c = fm.lib.fmoe_workspace_bytes(ctypes.byref(L), 1, 4, 64)
    assert 0 < a < b and a < c and a % 256 == 0
    # h for T tokens x (K+1) slots x I floats fits
    assert b >= 16 * 5 * 1024 * 4
    assert fm.lib.fmoe_workspace_bytes(ctypes.byref(L), 0, 4, 1) == 0


def test_batched_workspace_holds_outputs_and_plan(fm):
    L = fm.fmoe_layer()
    L.bits, L.group, L.hidden, L.inter, L.n_experts, L.has_shared = 4, 64, 4096, 1024, 512, 1
    b = fm.lib.fmoe_workspace_bytes(ctypes.byref(L), 16, 4, 1)
    h = 16 * 5 * 1024 * 4           # h  [T][K+S][I]
    y = 16 * 5 * 4096 * 4           # y  [T][K+S][H]
    plan = (8 + 8 * (16 * 4 + 16)) * 4   # header + one item per (token, slot) at worst
    assert b >= h + y + plan


def test_new_entry_points_check_arguments(fm):
    lib = fm.lib
    L = fm.fmoe_layer()
    L.bits, L.group, L.hidden, L.inter, L.n_experts, L.has_shared = 4, 64, 512, 128, 8, 0
    L.experts = 4096 * 16
    out = ctypes.c_void_p()
    assert lib.fmoe_ws_batch_plan(None, ctypes.byref(L), 2, 2, ctypes.byref(out)) == fm.ERR_INVALID_ARG
    assert lib.fmoe_ws_batch_plan(256, ctypes.byref(L), 0, 2, ctypes.byref(out)) == fm.ERR_INVALID_ARG
    assert lib.fmoe_ws_batch_plan(256, ctypes.byref(L), 2, 2, None) == fm.ERR_INVALID_ARG
    # a plan pointer inside the workspace, past its header
    assert lib.fmoe_ws_batch_plan(4096, ctypes.byref(L), 2, 2, ctypes.byref(out)) == fm.OK
    assert out.value > 4096 and out.value % 256 == 0
    # expert_ffn: T out of range, misaligned ids
    assert lib.fmoe_expert_ffn(ctypes.byref(L), 16, 17, 2, 16, 16, 256, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_expert_ffn(ctypes.byref(L), 2, 1, 2, 16, 16, 256, None) == fm.ERR_INVALID_ARG
    # no-alloc block: K > E, null input, misaligned output
    assert lib.fmoe_moe_block_noalloc(ctypes.byref(L), 16, 16, 16, 32, 9, None, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_moe_block_noalloc(ctypes.byref(L), None, 16, 16, 32, 2, None, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_moe_block_noalloc(ctypes.byref(L), 16, 16, 16, 40, 2, None, None) == fm.ERR_INVALID_ARG
    # router projection: null or misaligned matrix, T / E / H out of range, logits overlapping x
    assert lib.fmoe_router_logits(None, 4096, 1, 512, 8, 8192, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_router_logits(8, 4096, 1, 512, 8, 8192, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_router_logits(16, 4096, 17, 512, 8, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_router_logits(16, 4096, 1, 500, 8, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_router_logits(16, 4096, 1, 512, 0, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_router_logits(16, 1 << 20, 1, 512, 8, (1 << 20) + 64, None) == fm.ERR_INVALID_ARG
    # dense matrix rows: the record size is the oracle's, bad shapes are refused
    import oracle
    for bits in (4, 2):
        for H in (64, 192, 512, 2048, 4096, 8192):
            assert lib.fmoe_dense_row_bytes(bits, H) == oracle.dense_record_words(bits, H)[2] * 4
    assert lib.fmoe_dense_row_bytes(3, 512) == 0 and lib.fmoe_dense_row_bytes(4, 500) == 0
    # dense matvec: bad bits, T out of range, y overlapping x
    assert lib.fmoe_dense_gemv(16, 3, 8, 512, 4096, 1, None, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_dense_gemv(16, 4, 8, 512, 4096, 17, None, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_dense_gemv(16, 4, 8, 512, 4096, 1, None, 4096 + 64, None) == fm.ERR_INVALID_ARG
    # rmsnorm: T out of range, negative eps, x overlapping h without being h
    assert lib.fmoe_rmsnorm(4096, None, 0, 512, 1e-6, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_rmsnorm(4096, None, 1, 512, -1.0, 1 << 20, None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_rmsnorm(4096, None, 2, 512, 1e-6, 4096 + 64, None) == fm.ERR_INVALID_ARG
    # route from x: K > E, a gate pointer without the gate vector
    assert lib.fmoe_route_from_x(16, 4096, 1, 512, 8, 9, None, 1 << 20, 1 << 21, 1 << 22, None,
                                 None) == fm.ERR_INVALID_ARG
    assert lib.fmoe_route_from_x(16, 4096, 1, 512, 8, 2, None, 1 << 20, 1 << 21, 1 << 22, 1 << 23,
                                 None) == fm.ERR_INVALID_ARG
