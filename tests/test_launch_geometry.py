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
NAMES = ["fused_ok", "fused_grid", "fused_smem", "fused_ctrl", "xs_off", "part_off", "hbuf_off", "hb",
         "dscr_off", "darea_off", "darea_bytes", "ring_off", "nstage", "stage_bytes", "R", "nparts", "len_max",
         "batch_grid", "G", "gu_warps", "gu_rows", "gu_nstage", "gu_stage", "gu_xs", "gu_smem",
         "d_rows", "d_h", "d_smem", "batch_ctrl"]


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


def pieces(fm, bits, H, I, K, S, block, sms=SMS):
    out = (ctypes.c_int64 * 33)()
    assert fm.lib.fmoe_debug_block_pieces(bits, H, I, K, S, sms, block, out, 33) == fm.OK
    n = out[0]
    keys = ("slot", "i0", "cnt", "loc", "col_off", "sb_off", "g0", "ng")
    return [dict(zip(keys, out[1 + 8 * q: 9 + 8 * q])) for q in range(min(n, 4))], n


def parts(bits, H, I):
    p, _ = oracle.layout(bits, H, I)
    return p


SHAPES = list(itertools.product((4, 2), (64, 128, 192, 256, 512, 1024, 2048, 4096, 8192),
                                (64, 128, 320, 512, 1024, 2048, 4096), (1, 2, 4, 10, 16), (0, 1)))


@pytest.mark.parametrize("bits,H,I,K,S", SHAPES)
def test_geometry(fm, bits, H, I, K, S):
    g = geometry(fm, bits, H, I, K, S)
    p = parts(bits, H, I)
    gu_row, dcol, dsb = p["gate_q"][1], p["down_q"][1], p["down_sb"][1]
    # the batched path serves every shape the ABI accepts
    assert g["batch_grid"] == SMS
    assert 1 <= g["G"] <= 4 and g["gu_nstage"] >= 2
    assert g["gu_rows"] == 2 * g["gu_warps"] and I % g["gu_rows"] == 0
    assert g["gu_stage"] >= g["gu_rows"] * gu_row
    assert g["gu_xs"] >= g["G"] * 8 * (H // 32 + 1) * 16 + g["G"] * (H // 32) * 4
    assert g["gu_smem"] == g["batch_ctrl"] + g["gu_xs"] + g["gu_nstage"] * g["gu_stage"] <= SMEM_MAX
    assert (g["batch_ctrl"] + g["gu_xs"]) % 16 == 0 and g["gu_stage"] % 16 == 0
    assert g["d_rows"] == 32 * (32 // bits) and g["d_h"] >= g["G"] * I * 4
    assert g["d_smem"] <= SMEM_MAX
    if not g["fused_ok"]:
        # shapes the persistent kernel does not take (slice counts not powers of
        # two, or its regions do not fit) run on the batched path, checked above
        assert g["fused_smem"] == 0 or not (H // 32 & (H // 32 - 1) == 0)
        return
    NS = K + S
    assert g["fused_grid"] == SMS
    assert g["xs_off"] >= g["fused_ctrl"]
    assert g["part_off"] >= g["xs_off"] + H * 4
    assert g["hbuf_off"] >= g["part_off"] + 2 * g["nstage"] * g["R"] * g["nparts"] * 2 * 4
    assert g["hb"] >= (5 if bits == 4 else 9)
    assert g["len_max"] == -(-NS * I // SMS)
    assert g["dscr_off"] >= g["hbuf_off"] + g["len_max"] * g["hb"] * 4
    assert g["darea_off"] >= g["dscr_off"] + 8 * 128 * 4    # the down warps' transpose scratch
    assert g["ring_off"] >= g["darea_off"] + g["darea_bytes"]
    assert g["nstage"] >= 2 and g["stage_bytes"] >= g["R"] * gu_row
    assert g["fused_smem"] == g["ring_off"] + g["nstage"] * g["stage_bytes"] <= SMEM_MAX
    for k in ("xs_off", "part_off", "hbuf_off", "dscr_off", "darea_off", "darea_bytes", "ring_off", "stage_bytes"):
        assert g[k] % 128 == 0, k            # bulk-copy destinations: 16-byte aligned at least
    # every block's columns fit its down area, each copy 16-byte aligned
    covered = 0
    for c in range(SMS):
        pcs, n = pieces(fm, bits, H, I, K, S, c)
        assert n <= 4
        loc = 0
        for q in pcs:
            assert q["loc"] == loc and 0 <= q["slot"] < NS and 0 <= q["i0"] and q["i0"] + q["cnt"] <= I
            assert q["g0"] == q["i0"] // 64 and q["ng"] == (q["i0"] + q["cnt"] - 1) // 64 - q["g0"] + 1
            assert q["col_off"] % 128 == 0 and q["sb_off"] % 128 == 0
            assert q["sb_off"] >= q["col_off"] + q["cnt"] * dcol
            assert q["sb_off"] + q["ng"] * dsb <= g["darea_bytes"]
            assert (q["i0"] * dcol) % 16 == 0 and (q["cnt"] * dcol) % 16 == 0 and (q["ng"] * dsb) % 16 == 0
            loc += q["cnt"]
        covered += loc
    assert covered == NS * I


def test_pieces_cover_every_column_once(fm):
    for bits, H, I, K, S in ((4, 4096, 1024, 4, 1), (2, 4096, 1024, 4, 1), (4, 2048, 512, 10, 0),
                             (4, 512, 128, 2, 0), (4, 1024, 64, 1, 0)):
        seen = {}
        for c in range(SMS):
            pcs, _ = pieces(fm, bits, H, I, K, S, c)
            for q in pcs:
                for i in range(q["i0"], q["i0"] + q["cnt"]):
                    assert (q["slot"], i) not in seen
                    seen[(q["slot"], i)] = c
        assert len(seen) == (K + S) * I
        # a block's columns are consecutive in slot-major order
        order = sorted(seen, key=lambda si: si[0] * I + si[1])
        owners = [seen[k] for k in order]
        assert owners == sorted(owners)


def test_qwen_geometry_is_what_the_design_states(fm):
    g = geometry(fm, 4, 4096, 1024, 4, 1)
    assert g["fused_ok"] and g["R"] == 6 and g["stage_bytes"] == 6 * 4608 and g["fused_smem"] <= SMEM_MAX
    assert g["len_max"] == 35 and g["nstage"] >= 3
    assert (g["G"], g["gu_warps"], g["gu_nstage"], g["gu_stage"]) == (4, 8, 2, 16 * 4608)


def test_geometry_rejects_short_output(fm):
    out = (ctypes.c_int64 * 4)()
    assert fm.lib.fmoe_debug_launch_geometry(4, 512, 128, 2, 0, SMS, SMEM_MAX, out, 4) == fm.ERR_INVALID_ARG
    assert fm.lib.fmoe_debug_block_pieces(4, 512, 128, 2, 0, SMS, 0, out, 4) == fm.ERR_INVALID_ARG
    big = (ctypes.c_int64 * 33)()
    assert fm.lib.fmoe_debug_block_pieces(4, 512, 128, 2, 0, SMS, SMS, big, 33) == fm.ERR_INVALID_ARG
