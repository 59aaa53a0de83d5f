"""Host arithmetic of the launch geometry (no GPU): for every shape the ABI
accepts, the persistent kernel's and the batched kernels' shared-memory layouts
fit the device limit, keep their regions apart and aligned for bulk copies, and
the batched path exists (it serves every shape)."""
import ctypes
import itertools

import pytest

import oracle
from quantized_moe_expert_05_b300 import build

SMS, SMEM_MAX = 148, 232448          # B300: SMs, opt-in shared memory per block

# index names of the geometry vector (include/fmoe.h, FMOE_GEO_*)
NAMES = ["fused_ok", "fused_grid", "fused_smem", "fused_ctrl", "part_off", "stage_off", "hs_off", "hs_slot",
         "darea_off", "dslot", "ring_off", "nstage", "stage_bytes", "rows_per_stage", "nrmax", "nparts",
         "tail_rows", "batch_grid", "G", "gu_warps", "gu_rows", "gu_nstage", "gu_stage", "gu_xs", "gu_smem",
         "d_rows", "d_nstage", "d_stage", "d_xs", "d_smem", "batch_ctrl"]


@pytest.fixture(scope="module")
def fm():
    build.build()
    from quantized_moe_expert_05_b300 import fmoe
    return fmoe


def geometry(fm, bits, H, I, K, S, sms=SMS, smem=SMEM_MAX):
    out = (ctypes.c_int64 * len(NAMES))()
    st = fm.lib.fmoe_debug_launch_geometry(bits, H, I, K, S, sms, smem, out, len(NAMES))
    assert st == fm.OK
    return dict(zip(NAMES, out))


def records(bits, H, I):
    parts, _ = oracle.layout(bits, H, I)
    return parts["gate_q"][1], parts["down_q"][1]       # gate/up and down record strides


SHAPES = list(itertools.product((4, 2), (64, 128, 192, 256, 512, 1024, 2048, 4096, 8192),
                                (64, 128, 320, 512, 1024, 2048, 4096), (1, 2, 4, 10, 16), (0, 1)))


@pytest.mark.parametrize("bits,H,I,K,S", SHAPES)
def test_geometry(fm, bits, H, I, K, S):
    g = geometry(fm, bits, H, I, K, S)
    gu_row, d_row = records(bits, H, I)
    NS = K + S
    # the batched path serves every shape the ABI accepts
    assert g["batch_grid"] == SMS
    assert 1 <= g["G"] <= 4 and g["gu_nstage"] >= 2 and g["d_nstage"] >= 2
    assert g["gu_rows"] == 2 * g["gu_warps"] and I % g["gu_rows"] == 0 and H % g["d_rows"] == 0
    assert g["gu_stage"] >= g["gu_rows"] * gu_row and g["d_stage"] >= g["d_rows"] * d_row
    for pre in ("gu", "d"):
        cols = H if pre == "gu" else I
        assert g[pre + "_xs"] >= g["G"] * 8 * (cols // 32 + 1) * 16 + g["G"] * (cols // 32) * 4
        assert g[pre + "_smem"] == g["batch_ctrl"] + g[pre + "_xs"] + g[pre + "_nstage"] * g[pre + "_stage"]
        assert g[pre + "_smem"] <= SMEM_MAX
        assert (g["batch_ctrl"] + g[pre + "_xs"]) % 16 == 0 and g[pre + "_stage"] % 16 == 0
    if not g["fused_ok"]:
        # shapes the persistent kernel does not take (slice counts not powers of
        # two, or its regions do not fit) run on the batched path, checked above
        assert g["fused_smem"] == 0
        return
    ndmax = -(-H // SMS)
    nr_bytes = NS * g["nrmax"] * g["nparts"] * 2 * 4
    assert g["fused_grid"] == SMS
    assert g["part_off"] >= g["fused_ctrl"]
    assert g["stage_off"] >= g["part_off"] + nr_bytes
    assert g["hs_off"] >= g["stage_off"] + 2 * I * 8
    assert g["hs_slot"] >= 8 * (I // 32 + 1) * 16
    assert g["darea_off"] >= g["hs_off"] + max(NS * g["hs_slot"], H * 4)
    assert g["dslot"] >= ndmax * d_row
    assert g["ring_off"] >= g["darea_off"] + NS * g["dslot"]
    assert g["nstage"] >= 2 and g["stage_bytes"] >= g["rows_per_stage"] * gu_row
    assert g["fused_smem"] == g["ring_off"] + g["nstage"] * g["stage_bytes"] <= SMEM_MAX
    for k in ("part_off", "stage_off", "hs_off", "hs_slot", "darea_off", "dslot", "ring_off", "stage_bytes"):
        assert g[k] % 128 == 0, k            # bulk-copy destinations: 16-byte aligned at least
    assert ndmax <= g["tail_rows"]


def test_qwen_geometry_is_what_the_design_states(fm):
    g = geometry(fm, 4, 4096, 1024, 4, 1)
    assert g["fused_ok"] and g["nstage"] == 4 and g["stage_bytes"] == 6 * 4608 and g["fused_smem"] <= SMEM_MAX
    assert (g["G"], g["gu_warps"], g["gu_nstage"], g["gu_stage"]) == (4, 8, 2, 16 * 4608)
    assert (g["d_nstage"], g["d_stage"]) == (8, 32 * 576)


def test_geometry_rejects_short_output(fm):
    out = (ctypes.c_int64 * 4)()
    assert fm.lib.fmoe_debug_launch_geometry(4, 512, 128, 2, 0, SMS, SMEM_MAX, out, 4) == fm.ERR_INVALID_ARG
