"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Workloads: the tiny block (H 512, 8 experts, top-2), the Qwen-shaped block
(H 4096, 512 experts, top-4 + shared, I 1024) in 4-bit and 2-bit, the same
block at batch 1..16 with Zipf(1.1) routing, and the 48-layer stack (H 2048,
512 experts, top-10, I 512).  Expert ids must match exactly; outputs within
max relative error 2e-3 (both the max-normalised and the elementwise form).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from fmoe_testlib import (STACK_FLOOR, TOL, assert_close, gpu_pool, make_layer, oracle_block, oracle_expert,
                          oracle_pool, oracle_stack_token, rel_errors)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU only with -m gpu
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module")
def fm():
    from quantized_moe_expert_05_b300 import build
    build.build()
    from quantized_moe_expert_05_b300 import fmoe
    return fmoe


def run_block(fm, layer, shape, inp, K, ws):
    x = inp.x.cuda()
    lg = inp.logits.cuda()
    res = inp.residual.cuda()
    out = fm.moe_block(layer, x, lg, res, K, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    return out.cpu().numpy()


def check_block(fm, layer, shape, inp, K, ws, shared_index=0):
    got = run_block(fm, layer, shape, inp, K, ws)
    T = inp.x.shape[0]
    ref = oracle_block(shape, 0, inp.x.numpy(), inp.logits.numpy(), inp.residual.numpy(), K, shared_index)
    info = fm.ws_routing(ws, layer, T, K)
    ids = info["ids"].cpu().numpy()
    assert np.array_equal(ids, ref["ids"]), (ids, ref["ids"])
    assert_close(info["weights"].cpu().numpy(), ref["weights"], what="routing weights")
    if ref["gate"] is not None:
        assert_close(info["gate"].cpu().numpy(), ref["gate"], what="shared gate")
    errs = [assert_close(got[t], ref["out"][t], what=f"out token {t}") for t in range(T)]
    return max(e[0] for e in errs)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("E,K", [(8, 2), (8, 8), (5, 3), (33, 1), (512, 4), (512, 10), (1000, 16), (1024, 16)])
def test_route_matches_oracle(fm, E, K):
    g = torch.Generator().manual_seed(E * 100 + K)
    cases = [torch.randn((16, E), generator=g),
             torch.randint(-3, 4, (16, E), generator=g).float()]          # many ties
    z = torch.zeros((3, E))
    z[0, ::2] = -0.0
    z[1, : E // 2] = -0.0
    cases.append(z)                                                        # -0 == +0
    for lg in cases:
        ids, w = fm.route(lg.cuda(), K)
        torch.cuda.synchronize()
        for t in range(lg.shape[0]):
            rid, rw = oracle.route(lg[t].numpy(), K)
            assert ids[t].cpu().tolist() == rid.tolist(), (t, lg[t])
            assert_close(w[t].cpu().numpy(), rw, what="weights")


@pytest.mark.parametrize("T,E,H", [(1, 8, 512), (3, 100, 192), (1, 512, 4096), (5, 512, 4096), (16, 512, 4096),
                                   (16, 512, 2048), (2, 7, 256), (8, 37, 1024), (4, 1, 64)])
def test_router_projection_matches_oracle(fm, T, E, H):
    shape = dataclasses.replace(synth.TINY, hidden=H, n_experts=E)
    w = synth.router_matrix(shape, layer=T)
    x = synth.normal(7, T, (T, H))
    wsg = synth.shared_gate_vector(shape, layer=T)
    K = min(4, E)
    logits, ids, weights, gate = fm.route_from_x(w.cuda(), x.cuda(), K, wsg.cuda())
    torch.cuda.synchronize()
    ref = oracle.router_logits(w.numpy().view(np.uint16), x.numpy())
    got = logits.cpu().numpy()
    for t in range(T):
        assert_close(got[t], ref[t], what=f"logits token {t}")
        # the routing decision is taken on the GPU's own fp32 logits, so the
        # oracle routes those exactly
        rid, rw = oracle.route(got[t], K)
        assert ids[t].cpu().tolist() == rid.tolist()
        assert_close(weights[t].cpu().numpy(), rw, what="weights")
        assert_close(gate[t:t + 1].cpu().numpy(), [oracle.shared_gate(wsg.numpy().view(np.uint16), x[t].numpy())],
                     what="shared gate")
    # the projection alone writes the same logits, bit for bit (fixed summation order)
    again = fm.router_logits(w.cuda(), x.cuda())
    torch.cuda.synchronize()
    assert torch.equal(again.cpu(), logits.cpu())


@pytest.mark.parametrize("bits,N,H,T", [(4, 4096, 4096, 1), (4, 4096, 4096, 16), (2, 192, 512, 3), (4, 1000, 2048, 5),
                                         (2, 2048, 2048, 1), (4, 101, 320, 2), (2, 67, 192, 7), (4, 33, 64, 16)])
def test_dense_gemv_matches_oracle(fm, bits, N, H, T):
    w = synth.dense_matrix(N, H, bits, seed=9, tag=bits * 100 + T)
    x = synth.normal(9, 10 + T, (T, H))
    res = synth.normal(9, 20 + T, (T, N))
    W = oracle.dense_weights(w.numpy().view(np.uint32), bits, N, H)
    ref = oracle.dense_matvec(W, x.numpy(), res.numpy())
    wd = w.cuda()
    y = fm.dense_gemv(wd, bits, N, x.cuda(), residual=res.cuda())
    torch.cuda.synchronize()
    for t in range(T):
        assert_close(y[t].cpu().numpy(), ref[t], what=f"o_proj token {t}")
    # in place: residual and output the same buffer, and bit for bit the same result
    y2 = res.cuda()
    fm.dense_gemv(wd, bits, N, x.cuda(), residual=y2, y=y2)
    torch.cuda.synchronize()
    assert torch.equal(y2.cpu(), y.cpu())


@pytest.mark.parametrize("T,H", [(1, 4096), (16, 4096), (3, 2048), (2, 192)])
def test_rmsnorm_weight_matches_oracle(fm, T, H):
    h = synth.normal(11, T, (T, H)) * 3.0
    wn = synth.norm_weight(H, 11, T)
    x = fm.rmsnorm(h.cuda(), 1e-6, wn.cuda())
    torch.cuda.synchronize()
    for t in range(T):
        assert_close(x[t].cpu().numpy(), oracle.rms_norm(h[t].numpy(), 1e-6, wn.numpy()), what=f"rmsnorm token {t}")
    hd = h.cuda()
    fm.rmsnorm(hd, 1e-6, wn.cuda(), x=hd)            # in place
    torch.cuda.synchronize()
    assert torch.equal(hd.cpu(), x.cpu())


def test_slot_pool_zipf_routing_matches_oracle(fm):
    """A quarter of the experts in HBM slots, the rest copied in from pinned
    host memory as the routing asks (Zipf(1.1) popularity); the block runs
    against the slots with logits remapped to them.  Ids (mapped back from
    slots) exact, outputs within 2e-3 of the oracle on the full expert set, at
    T = 1 (single launch) and T = 4 (batched path)."""
    shape = dataclasses.replace(synth.QWEN_Q4, name="pool_h1024_e64_top4_shared_i512_q4", hidden=1024, inter=512,
                                n_experts=64)
    K, S = shape.top_k, 16
    nw = synth.blob_bytes(shape.bits, shape.hidden, shape.inter) // 4
    host = torch.empty(shape.n_experts * nw, dtype=torch.int32, pin_memory=True)
    host.copy_(gpu_pool(shape, 0, shape.n_experts).cpu())
    slots = torch.zeros(S * nw, dtype=torch.int32, device="cuda")
    shared = gpu_pool(shape, 0, 1, first=shape.n_experts)
    wsg = synth.shared_gate_vector(shape, 0).cuda()
    pool = fm.SlotPool(S, shape.n_experts, nw * 4, slots.data_ptr(), host.data_ptr())
    layer = fm.Layer(shape.bits, shape.hidden, shape.inter, S, slots, shared, wsg)
    copy = torch.cuda.Stream()
    step = 0
    for T, n_steps in ((1, 12), (4, 4)):
        ws = fm.new_workspace(layer, T, K)
        for _ in range(n_steps):
            step += 1
            logits = synth.zipf_logits(shape.seed, 500 + step, T, shape.n_experts, 1.1)
            x = synth.normal(shape.seed, 600 + step, (T, shape.hidden))
            res = synth.normal(shape.seed, 700 + step, (T, shape.hidden))
            ids_dev, _ = fm.route(logits.cuda(), K)
            ids = ids_dev.cpu().numpy()
            sl_of, loads = pool.plan(ids.flatten().tolist(), keep=0)
            pool.load(loads, stream=copy)
            done = torch.cuda.Event()
            done.record(copy)
            torch.cuda.current_stream().wait_event(done)
            slot_ids = np.array(sl_of, dtype=np.int32).reshape(T, K)
            slot_logits = torch.from_numpy(pool.slot_logits(logits.numpy(), ids, slot_ids)).cuda()
            out = fm.moe_block(layer, x.cuda(), slot_logits, res.cuda(), K, ws)
            torch.cuda.synchronize()
            assert fm.last_device_error(ws) == fm.OK
            expert_of = {int(sl): int(e) for e, sl in zip(ids.flatten(), sl_of)}
            got_slots = fm.ws_routing(ws, layer, T, K)["ids"].cpu().numpy()
            for t in range(T):
                ref = oracle_block(shape, 0, x[t:t + 1].numpy(), logits[t:t + 1].numpy(), res[t:t + 1].numpy(), K)
                assert [expert_of[int(v)] for v in got_slots[t]] == list(ref["ids"][0]), (step, t)
                assert_close(out[t].cpu().numpy(), ref["out"][0], what=f"pool step {step} token {t}")
    st = pool.stats()
    assert st["misses"] > S and st["hits"] > 0, st


# ---------------------------------------------------------------------------
# tiny block (every output, several draws, fused single-launch path)
# ---------------------------------------------------------------------------
def test_tiny_block_all_outputs(fm):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 16, shape.top_k)
    for tag in range(6):
        inp = synth.block_inputs(shape, 1, tag=tag)
        check_block(fm, layer, shape, inp, shape.top_k, ws)


@pytest.mark.parametrize("K", [1, 2, 8])
def test_tiny_block_k_extremes(fm, K):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 16, K)
    for T in (1, 3, 16):
        inp = synth.block_inputs(shape, T, tag=7 + T)
        check_block(fm, layer, shape, inp, K, ws)


def test_tiny_block_ties_and_signed_zero(fm):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 1, 2)
    inp = synth.block_inputs(shape, 1, tag=20)
    inp.logits[:] = torch.tensor([[0.5, -0.0, 0.5, 0.0, 0.5, -1.0, 0.25, 0.5]])
    check_block(fm, layer, shape, inp, 2, ws)
    inp.logits[:] = torch.tensor([[-0.0, -1.0, 0.0, -2.0, -0.0, -3.0, -1.0, -0.0]])
    check_block(fm, layer, shape, inp, 2, ws)


def test_expert_ffn_tiny_and_qwen(fm):
    for shape, T, K in ((synth.TINY, 3, 2), (synth.QWEN_Q4, 2, 4)):
        layer = make_layer(fm, shape)
        ws = fm.new_workspace(layer, T, K)
        g = torch.Generator().manual_seed(5)
        ids = torch.stack([torch.randperm(shape.n_experts, generator=g)[:K] for _ in range(T)]).int()
        x = synth.normal(shape.seed, 77, (T, shape.hidden))
        y = fm.expert_ffn(layer, ids.cuda(), x.cuda(), ws)
        torch.cuda.synchronize()
        assert fm.last_device_error(ws) == fm.OK
        y = y.cpu().numpy()
        for t in range(T):
            for k in range(K):
                ref = oracle.expert_ffn(oracle_expert(shape, 0, int(ids[t, k])), x[t].numpy())
                assert_close(y[t, k], ref, what=f"y[{t},{k}]")
            if shape.has_shared:
                ref = oracle.expert_ffn(oracle_expert(shape, 0, shape.n_experts), x[t].numpy())
                assert_close(y[t, K], ref, what=f"shared y[{t}]")


def test_expert_ffn_bad_id_is_reported_not_faulted(fm):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 1, 2)
    ids = torch.tensor([[1, 99]], dtype=torch.int32, device="cuda")
    x = synth.normal(0, 5, (1, shape.hidden)).cuda()
    y = fm.expert_ffn(layer, ids, x, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.ERR_INVALID_ARG
    assert torch.all(y[0, 1] == 0)
    # the context is still usable and the error word was cleared
    y = fm.expert_ffn(layer, ids[:, :1].contiguous(), x, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK


def test_zero_weight_invariance_on_gpu(fm):
    shape = synth.TINY
    pool = gpu_pool(shape, 0, shape.n_experts)
    layer = make_layer(fm, shape, pool=pool)
    ws = fm.new_workspace(layer, 1, 3)
    inp = synth.block_inputs(shape, 1, tag=30)
    inp.logits[0] = torch.tensor([1.0, 0.5, 1.0 - 1e4, -2e4, -2e4, -2e4, -2e4, -2e4])
    a = run_block(fm, layer, shape, inp, 3, ws)
    nw = pool.numel() // shape.n_experts
    pool2 = pool.clone()
    pool2[2 * nw:3 * nw] = torch.randint(-2 ** 31, 2 ** 31 - 1, (nw,), dtype=torch.int32, device="cuda") & 0x0F0F0F0F
    b = run_block(fm, make_layer(fm, shape, pool=pool2), shape, inp, 3, ws)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("T", [1, 3])
def test_poisoned_outputs_and_scratch_are_fully_written(fm, T):
    """Every output element and every scratch word a call reads is written by
    the call: outputs and the whole workspace past its state (the 256-byte
    header and the single-launch kernel's accumulators, 256 + 24*H bytes
    rounded up to 256) start as NaN."""
    shape = synth.BlockShape("tiny_shared_h512_e8_top2_i128_q4", 512, 128, 8, 2, True, 4, 0.002, 0.02, -0.1,
                             0.0, seed=23)
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 3, 2)
    state = (256 + 24 * shape.hidden + 255) // 256 * 256
    ws[state:].view(torch.float32).fill_(float("nan"))
    inp = synth.block_inputs(shape, T, tag=90)
    out = torch.full((T, shape.hidden), float("nan"), device="cuda")
    fm.moe_block(layer, inp.x.cuda(), inp.logits.cuda(), inp.residual.cuda(), 2, ws, out=out)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    assert torch.isfinite(out).all()
    ref = oracle_block(shape, 0, inp.x.numpy(), inp.logits.numpy(), inp.residual.numpy(), 2)
    got = out.cpu().numpy()
    for t in range(T):
        assert_close(got[t], ref["out"][t], what=f"poisoned run, token {t}")

    ws[state:].view(torch.float32).fill_(float("nan"))
    ids = torch.tensor([[1, 5], [5, 1], [0, 7]][:T], dtype=torch.int32, device="cuda")
    y = torch.full((T, 3, shape.hidden), float("nan"), device="cuda")
    fm.expert_ffn(layer, ids, inp.x.cuda(), ws, y=y)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    assert torch.isfinite(y).all()


def test_out_aliases_residual(fm):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 1, 2)
    inp = synth.block_inputs(shape, 1, tag=40)
    ref = oracle_block(shape, 0, inp.x.numpy(), inp.logits.numpy(), inp.residual.numpy(), 2)
    res = inp.residual.cuda()
    fm.moe_block(layer, inp.x.cuda(), inp.logits.cuda(), res, 2, ws, out=res)
    torch.cuda.synchronize()
    assert_close(res.cpu().numpy()[0], ref["out"][0], what="in-place out")


def test_ragged_shape_general_path(fm):
    # H and I that are not powers of two: 6 and 10 lane slices per row
    shape = synth.BlockShape("ragged_h192_e6_top3_i320_q4", 192, 320, 6, 3, True, 4,
                             0.002, 0.02, -0.1, 0.0, seed=11)
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 5, 3)
    for T in (1, 5):
        check_block(fm, layer, shape, synth.block_inputs(shape, T, tag=T), 3, ws)
    shape2 = synth.BlockShape("ragged_h192_e6_top3_i320_q2", 192, 320, 6, 3, True, 2,
                              0.01, 0.05, -0.1, 0.0, seed=12)
    layer2 = make_layer(fm, shape2)
    check_block(fm, layer2, shape2, synth.block_inputs(shape2, 2, tag=1), 3, ws)


# ---------------------------------------------------------------------------
# Qwen-shaped block, 4-bit and 2-bit, full size
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def qwen_pools():
    return {s.name: gpu_pool(s, 0, s.n_experts) for s in (synth.QWEN_Q4, synth.QWEN_Q2)}


@pytest.mark.parametrize("shape", [synth.QWEN_Q4, synth.QWEN_Q2], ids=lambda s: s.name)
def test_qwen_block_batch1(fm, qwen_pools, shape):
    layer = make_layer(fm, shape, pool=qwen_pools[shape.name])
    ws = fm.new_workspace(layer, 1, 4)
    worst = 0.0
    for tag in range(3):
        worst = max(worst, check_block(fm, layer, shape, synth.block_inputs(shape, 1, tag=tag), 4, ws))
    print(f"{shape.name}: worst max-rel err {worst:.2e}")


def test_qwen_block_graph_replay_matches_eager(fm, qwen_pools):
    shape = synth.QWEN_Q4
    layer = make_layer(fm, shape, pool=qwen_pools[shape.name])
    ws = fm.new_workspace(layer, 1, 4)
    inp = synth.block_inputs(shape, 1, tag=5)
    x, lg, res = inp.x.cuda(), inp.logits.cuda(), inp.residual.cuda()
    eager = fm.moe_block(layer, x, lg, res, 4, ws).clone()
    out = torch.empty_like(res)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fm.moe_block(layer, x, lg, res, 4, ws, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fm.moe_block(layer, x, lg, res, 4, ws, out=out)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


# ---------------------------------------------------------------------------
# batch 1..16 with Zipf routing (unique experts read once)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_qwen_batch_zipf(fm, qwen_pools, T):
    shape = synth.QWEN_Q4_BATCH
    layer = make_layer(fm, shape, pool=_zipf_pool(shape))
    ws = fm.new_workspace(layer, 16, 4)
    check_block(fm, layer, shape, synth.block_inputs(shape, T, tag=T), 4, ws)


def check_plan(fm, layer, ws, T, K, ids, S):
    """The batch plan lists each distinct expert once (ceil(m/4) items for m
    tokens), covers every (token, slot) exactly once, tokens ascending."""
    plan = fm.ws_batch_plan(ws, layer, T, K)
    ids = np.asarray(ids)
    distinct = sorted(set(int(v) for v in ids.ravel()))
    assert plan["n_unique"] == len(distinct) + S
    seen, order = {}, []
    for expert, pairs in plan["items"]:
        assert 1 <= len(pairs) <= 4
        for t, k in pairs:
            assert (t, k) not in seen
            seen[(t, k)] = expert
            assert expert == (int(ids[t, k]) if k < K else -1)
        if not order or order[-1][0] != expert:
            order.append((expert, []))
        order[-1][1].extend(t for t, _ in pairs)
    want = {(t, k) for t in range(T) for k in range(K)} | ({(t, K) for t in range(T)} if S else set())
    assert set(seen) == want
    experts_in_order = [e for e, _ in order]
    assert len(experts_in_order) == len(set(experts_in_order)), "an expert's items are not contiguous"
    for _, toks in order:
        assert toks == sorted(toks)
    m = {e: sum(1 for v in seen.values() if v == e) for e in set(seen.values())}
    assert plan["n_items"] == sum((c + 3) // 4 for c in m.values())
    return plan


@pytest.mark.parametrize("T", [2, 16])
def test_batch_plan_reads_each_expert_once(fm, qwen_pools, T):
    shape = synth.QWEN_Q4_BATCH
    layer = make_layer(fm, shape, pool=_zipf_pool(shape))
    ws = fm.new_workspace(layer, 16, 4)
    inp = synth.block_inputs(shape, T, tag=T)
    run_block(fm, layer, shape, inp, 4, ws)
    ids = fm.ws_routing(ws, layer, T, 4)["ids"].cpu().numpy()
    plan = check_plan(fm, layer, ws, T, 4, ids, 1)
    print(f"T={T}: {plan['n_unique']} distinct experts (incl. shared) for {T * 4 + T} picks")


def test_batch_all_tokens_share_experts(fm, qwen_pools):
    # every token routes to the same 4 experts: 5 distinct experts, 4 items each
    shape = synth.QWEN_Q4_BATCH
    layer = make_layer(fm, shape, pool=_zipf_pool(shape))
    ws = fm.new_workspace(layer, 16, 4)
    inp = synth.block_inputs(shape, 16, tag=60)
    inp.logits[:] = inp.logits[0:1]
    check_block(fm, layer, shape, inp, 4, ws)
    plan = check_plan(fm, layer, ws, 16, 4, fm.ws_routing(ws, layer, 16, 4)["ids"].cpu().numpy(), 1)
    assert plan["n_unique"] == 5 and plan["n_items"] == 20


def test_batch_q2_zipf(fm, qwen_pools):
    shape = dataclasses.replace(synth.QWEN_Q2, zipf_s=1.1)
    layer = make_layer(fm, shape, pool=qwen_pools[synth.QWEN_Q2.name])
    ws = fm.new_workspace(layer, 8, 4)
    check_block(fm, layer, shape, synth.block_inputs(shape, 8, tag=3), 4, ws)


def test_expert_ffn_duplicate_ids(fm):
    # the same expert twice in one token and across tokens; the tiny block
    shape = synth.TINY
    layer = make_layer(fm, shape)
    T, K = 6, 3
    ws = fm.new_workspace(layer, T, K)
    ids = torch.tensor([[3, 3, 1], [1, 3, 0], [7, 7, 7], [0, 1, 3], [3, 5, 1], [1, 3, 3]], dtype=torch.int32)
    x = synth.normal(shape.seed, 78, (T, shape.hidden))
    y = fm.expert_ffn(layer, ids.cuda(), x.cuda(), ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    y = y.cpu().numpy()
    for t in range(T):
        for k in range(K):
            ref = oracle.expert_ffn(oracle_expert(shape, 0, int(ids[t, k])), x[t].numpy())
            assert_close(y[t, k], ref, what=f"y[{t},{k}]")
    check_plan(fm, layer, ws, T, K, ids.numpy(), 0)


_ZP = {}


def _zipf_pool(shape):
    if shape.name not in _ZP:
        _ZP[shape.name] = gpu_pool(shape, 0, shape.n_experts)
    return _ZP[shape.name]


# ---------------------------------------------------------------------------
# stacks
# ---------------------------------------------------------------------------
def _oracle_stack(shape, h0, logits, K, shared=False):
    return oracle.stack_decode(lambda l, e: oracle_expert(shape, l, e), h0, logits, K, shape.eps,
                               (lambda l: oracle_expert(shape, l, shape.n_experts)) if shared else None,
                               (lambda l: synth.shared_gate_vector(shape, l).numpy().view(np.uint16))
                               if shared else None)


@pytest.mark.parametrize("L", [1, 2, 5, 70])
def test_tiny_stack(fm, L):
    shape = synth.BlockShape("tiny_stack", 512, 128, 8, 2, True, 4, 0.002, 0.02, -0.1, 0.0, seed=21,
                             n_layers=L)
    layers = [make_layer(fm, shape, layer=l) for l in range(L)]
    ws = fm.new_workspace(layers[0], 1, 2, L)
    h0, logits = synth.stack_inputs(shape, 1)
    h = h0[0].clone().cuda()
    fm.stack_decode(layers, logits[0].cuda(), h, 2, shape.eps, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    ref, _ = _oracle_stack(shape, h0[0].numpy(), logits[0].numpy(), 2, shared=True)
    assert_close(h.cpu().numpy(), ref, what=f"tiny stack L={L}")


@pytest.fixture(scope="module")
def stack48_layers(fm):
    shape = synth.STACK48
    return [make_layer(fm, shape, layer=l) for l in range(shape.n_layers)]


def test_stack48_tokens(fm, stack48_layers):
    """The first 8 tokens of the 48-layer stack (H 2048, 512 experts per layer,
    top-10, I 512) through all 48 layers: ids of every layer exact, h within
    the tolerance.  The oracle runs in a spawned process pool."""
    shape = synth.STACK48
    T = 8
    ws = fm.new_workspace(stack48_layers[0], 1, shape.top_k, shape.n_layers)
    h0, logits = synth.stack_inputs(shape, T)
    with oracle_pool() as pool:
        futs = [pool.submit(oracle_stack_token, shape, h0[t].numpy(), logits[t].numpy(), shape.top_k)
                for t in range(T)]
        for t in range(T):
            h = h0[t].clone().cuda()
            fm.stack_decode(stack48_layers, logits[t].cuda(), h, shape.top_k, shape.eps, ws)
            torch.cuda.synchronize()
            assert fm.last_device_error(ws) == fm.OK
            got_ids = fm.ws_routing(ws, stack48_layers[0], shape.n_layers, shape.top_k)["ids"].cpu().numpy()
            ref, ids = futs[t].result()
            assert np.array_equal(got_ids, np.asarray(ids)), f"token {t}: routing differs"
            assert_close(h.cpu().numpy(), ref, what=f"stack48 token {t}", floor=STACK_FLOOR)


def test_ragged_stack_general_path(fm):
    """A stack whose shape the single-launch kernel does not take (H/32 = 6
    slices) runs per layer on the general path (RMSNorm launch + batched
    block), against the oracle."""
    shape = synth.BlockShape("ragged_stack_h192_e6_top3_i320_q4", 192, 320, 6, 3, True, 4, 0.002, 0.02, -0.1,
                             0.0, seed=41, n_layers=3)
    layers = [make_layer(fm, shape, layer=l) for l in range(shape.n_layers)]
    ws = fm.new_workspace(layers[0], 1, shape.top_k, shape.n_layers)
    h0, logits = synth.stack_inputs(shape, 2)
    for t in range(2):
        h = h0[t].clone().cuda()
        fm.stack_decode(layers, logits[t].cuda(), h, shape.top_k, shape.eps, ws)
        torch.cuda.synchronize()
        assert fm.last_device_error(ws) == fm.OK
        ref, ids = oracle_stack_token(shape, h0[t].numpy(), logits[t].numpy(), shape.top_k, shared=True)
        got_ids = fm.ws_routing(ws, layers[0], shape.n_layers, shape.top_k)["ids"].cpu().numpy()
        assert np.array_equal(got_ids, np.asarray(ids))
        assert_close(h.cpu().numpy(), ref, what=f"ragged stack token {t}")


# ---------------------------------------------------------------------------
# the bench's launch: a chain of Qwen-shaped blocks in one persistent launch
# (one routed pool for every block, each block its own shared expert and gate)
# ---------------------------------------------------------------------------
def _qwen_chain_layers(fm, shape, n, pool):
    nw = synth.blob_bytes(shape.bits, shape.hidden, shape.inter) // 4
    shared = torch.empty(n * nw, dtype=torch.int32, device="cuda")
    synth.fill_pool(shared, shape, 0, shape.n_experts, n)
    return [fm.Layer(shape.bits, shape.hidden, shape.inter, shape.n_experts, pool, shared[l * nw:(l + 1) * nw],
                     synth.shared_gate_vector(shape, l).cuda()) for l in range(n)]


def _oracle_chain(shape, h0, logits):
    """The chain as the oracle computes it: block l uses routed experts of the
    common pool and shared expert n_experts + l with gate vector l."""
    return oracle.stack_decode(lambda l, e: oracle_expert(shape, 0, e), h0, logits, shape.top_k, shape.eps,
                               lambda l: oracle_expert(shape, 0, shape.n_experts + l),
                               lambda l: synth.shared_gate_vector(shape, l).numpy().view(np.uint16))


@pytest.mark.parametrize("shape", [synth.QWEN_Q4, synth.QWEN_Q2], ids=lambda s: s.name)
def test_qwen_chain_as_benched(fm, qwen_pools, shape):
    """Four chained Qwen blocks (4-bit and 2-bit) against the oracle; then the
    64-block launch the bench times equals sixteen 4-block launches bit for
    bit (every block runs the same code on the same input whichever launch it
    is in, and the blocks' partial sums are added in exact integer arithmetic)."""
    import dataclasses
    n = 64
    layers = _qwen_chain_layers(fm, shape, n, qwen_pools[shape.name])
    h0, logits = synth.stack_inputs(dataclasses.replace(shape, n_layers=n), 1)
    ws = fm.new_workspace(layers[0], 1, shape.top_k, n)
    h4 = h0[0].clone().cuda()
    fm.stack_decode(layers[:4], logits[0, :4].contiguous().cuda(), h4, shape.top_k, shape.eps, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    ref, ids = _oracle_chain(dataclasses.replace(shape, n_layers=4), h0[0].numpy(), logits[0, :4].numpy())
    assert_close(h4.cpu().numpy(), ref, what=f"4-block chain {shape.name}")
    got_ids = fm.ws_routing(ws, layers[0], 4, shape.top_k)["ids"].cpu().numpy()
    assert np.array_equal(got_ids, np.asarray(ids)), (got_ids, ids)

    whole = h0[0].clone().cuda()
    fm.stack_decode(layers, logits[0].cuda(), whole, shape.top_k, shape.eps, ws)
    parts = h0[0].clone().cuda()
    for l0 in range(0, n, 4):
        fm.stack_decode(layers[l0:l0 + 4], logits[0, l0:l0 + 4].contiguous().cuda(), parts, shape.top_k,
                        shape.eps, ws)
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    assert torch.equal(whole, parts)
    assert torch.isfinite(whole).all()


def test_generator_cpu_gpu_identical():
    for shape, e in ((synth.QWEN_Q4, 7), (synth.QWEN_Q2, 300), (synth.STACK48, 511)):
        a = synth.expert_blob(shape, 3, e, device="cpu")
        b = synth.expert_blob(shape, 3, e, device="cuda").cpu()
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# bounded device-side waits
# ---------------------------------------------------------------------------
def test_bounded_wait_times_out_and_reports(fm):
    shape = synth.TINY
    layer = make_layer(fm, shape)
    ws = fm.new_workspace(layer, 1, 2)
    fm.debug_wait_test(ws, 8, 8, 1_000_000)          # all arrive: completes
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.OK
    fm.debug_wait_test(ws, 4, 5, 20_000)             # one arrival short: 20 ms time-out
    torch.cuda.synchronize()
    assert fm.last_device_error(ws) == fm.ERR_TIMEOUT
    assert fm.last_device_error(ws) == fm.OK         # cleared
    # the context stays usable
    check_block(fm, layer, shape, synth.block_inputs(shape, 1, tag=3), 2, fm.new_workspace(layer, 1, 2))
