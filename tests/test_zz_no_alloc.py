"""fmoe_moe_block_noalloc: the single-token block without a caller workspace.

This entry point serves callers that cannot allocate device memory, for
example code that runs inside an allocator or memory-pool callback, a plugin
whose host framework owns every device allocation, or a real-time loop that
must not block in cudaMalloc.  It keeps its scratch in a fixed array inside
the library instead of a workspace.  These tests call it through the C ABI
and check two calls in a row against fmoe_moe_block (with a workspace) and
against the fp64 oracle, at the tiny, a small, the Qwen-shaped 4-bit and the
48-layer stack's block shapes, and with shapes of different K and
intermediate size alternating from call to call (the array keeps the last
call's contents).

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import synth
from fmoe_testlib import TOL, assert_close, make_layer, oracle_block

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU only with -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module")
def fm():
    from quantized_moe_expert_05_b300 import build
    build.build()
    from quantized_moe_expert_05_b300 import fmoe
    return fmoe


SHARED_SMALL = synth.BlockShape("small_h1024_e16_top4_shared_i256_q4", 1024, 256, 16, 4, True, 4,
                                0.002, 0.02, -0.1, 0.0, seed=31)
SHARED_SMALL_Q2 = synth.BlockShape("small_h1024_e16_top4_shared_i256_q2", 1024, 256, 16, 4, True, 2,
                                   0.01, 0.05, -0.1, 0.0, seed=32)


@pytest.mark.parametrize("shape", [synth.TINY, SHARED_SMALL, SHARED_SMALL_Q2], ids=lambda s: s.name)
def test_noalloc_matches_workspace_call_twice(fm, shape):
    layer = make_layer(fm, shape)
    K = shape.top_k
    ws = fm.new_workspace(layer, 1, K)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for tag in (0, 1):                                   # two calls in a row
        inp = synth.block_inputs(shape, 1, tag=100 + tag)
        x, lg, res = inp.x.cuda(), inp.logits.cuda(), inp.residual.cuda()
        want = fm.moe_block(layer, x, lg, res, K, ws)
        got = fm.moe_block_noalloc(layer, x, lg, res, K, device_error=err)
        torch.cuda.synchronize()
        assert fm.last_device_error(ws) == fm.OK
        assert int(err.item()) == 0, "device-side error word of the scratch-free call"
        assert_close(got.cpu().numpy()[0], want.cpu().numpy()[0], tol=TOL, what=f"{shape.name} call {tag}")


def _check_against_oracle(fm, layer, shape, tag, err):
    inp = synth.block_inputs(shape, 1, tag=tag)
    got = fm.moe_block_noalloc(layer, inp.x.cuda(), inp.logits.cuda(), inp.residual.cuda(), shape.top_k,
                               device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device-side error word of the scratch-free call"
    ref = oracle_block(shape, 0, inp.x.numpy(), inp.logits.numpy(), inp.residual.numpy(), shape.top_k)
    assert_close(got.cpu().numpy()[0], ref["out"][0], what=f"{shape.name} tag {tag} against the oracle")


STACK_BLOCK = synth.BlockShape("stack_block_h2048_e512_top10_i512_q4", 2048, 512, 512, 10, False, 4,
                               0.002, 0.02, -0.1, 0.0, seed=4)


@pytest.mark.parametrize("shape", [synth.QWEN_Q4, STACK_BLOCK], ids=lambda s: s.name)
def test_noalloc_matches_oracle_at_full_size(fm, shape):
    layer = make_layer(fm, shape)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for tag in (200, 201):                               # two calls in a row
        _check_against_oracle(fm, layer, shape, tag, err)


def test_noalloc_alternating_shapes(fm):
    """Calls with different K and intermediate size in a row: nothing a call
    leaves in the shared array changes the next call's result."""
    shapes = [synth.TINY, synth.QWEN_Q4, SHARED_SMALL, synth.TINY, synth.QWEN_Q4]
    layers = {}
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for i, shape in enumerate(shapes):
        if shape.name not in layers:
            layers[shape.name] = make_layer(fm, shape)
        _check_against_oracle(fm, layers[shape.name], shape, 300 + i, err)


def test_noalloc_in_place_and_without_error_output(fm):
    shape = SHARED_SMALL
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 1, shape.top_k)
    inp = synth.block_inputs(shape, 1, tag=7)
    x, lg = inp.x.cuda(), inp.logits.cuda()
    want = fm.moe_block(layer, x, lg, inp.residual.cuda(), shape.top_k, ws)
    res = inp.residual.cuda()
    fm.moe_block_noalloc(layer, x, lg, res, shape.top_k, out=res)     # out aliases residual
    torch.cuda.synchronize()
    assert_close(res.cpu().numpy()[0], want.cpu().numpy()[0], what="in place")


def test_noalloc_rejects_shapes_beyond_its_scratch(fm):
    # H 8192 needs 256 + 24 * 8192 = 196,864 bytes of scratch, more than the
    # library's fixed 128 KiB array: refused up front.
    dummy = torch.zeros(1024, dtype=torch.int32, device="cuda")
    wsg = torch.zeros(8192, dtype=torch.int16, device="cuda")
    layer = fm.Layer(4, 8192, 4096, 64, dummy, dummy, wsg)
    x = torch.zeros((1, 8192), device="cuda")
    lg = torch.zeros((1, 64), device="cuda")
    with pytest.raises(fm.FmoeError) as e:
        fm.moe_block_noalloc(layer, x, lg, x.clone(), 16)
    assert e.value.status == fm.ERR_INVALID_ARG
    assert fm.workspace_bytes(layer, 1, 16) > fm.NOALLOC_SCRATCH_BYTES
