"""The seeded input generator: determinism, independence of chunking, ranges."""
import numpy as np
import torch

import synth


def test_blob_is_deterministic_and_chunk_independent():
    s = synth.TINY
    one = synth.expert_blob(s, 0, 5)
    many = synth.expert_blobs(s, 0, [3, 4, 5, 6])
    assert torch.equal(one, many[2])
    pool = torch.zeros(8 * one.numel(), dtype=torch.int32)
    synth.fill_pool(pool, s, 0, 0, 8, chunk=3)
    assert torch.equal(pool.view(8, -1)[5], one)
    assert not torch.equal(many[0], many[1])
    # another layer or seed gives other words
    assert not torch.equal(synth.expert_blob(s, 1, 5), one)
    assert not torch.equal(synth.expert_blob(s, 0, 5, seed=9), one)


def test_codes_uniform_and_scales_in_range():
    s = synth.QWEN_Q4
    blob = synth.expert_blob(s, 0, 17).numpy().view(np.uint32)
    parts, nbytes = synth.row_layout(s.bits, s.hidden, s.inter)
    assert blob.size * 4 == nbytes == 7077888
    base, stride = parts["gate_q"]
    rows = blob[: s.inter * stride // 4].reshape(s.inter, stride // 4)
    q = rows[:, base // 4: base // 4 + s.hidden // 8].astype(np.uint64).reshape(-1)
    nib = np.concatenate([(q >> np.uint64(4 * i)) & np.uint64(15) for i in range(8)])
    hist = np.bincount(nib.astype(np.int64), minlength=16) / nib.size
    assert np.all(np.abs(hist - 1 / 16) < 0.002)
    base, stride = parts["gate_sb"]
    sbw = rows[:, base // 4: base // 4 + s.hidden // 64].reshape(-1)
    sc = ((sbw & 0xFFFF).astype(np.uint32) << 16).view(np.float32)
    bi = ((sbw >> 16).astype(np.uint32) << 16).view(np.float32)
    assert sc.min() >= 0.0019 and sc.max() <= 0.0201
    assert bi.min() >= -0.1005 and bi.max() <= 0.0


def test_zipf_logits_popularity():
    l = synth.zipf_logits(3, 1, 2000, 512, 1.1)
    top = torch.topk(l, 4, dim=1).indices.flatten()
    counts = torch.bincount(top, minlength=512).sort(descending=True).values
    # the most popular expert is picked far more often than the median one
    assert counts[0] > 20 * max(int(counts[256]), 1)


def test_activations_deterministic():
    a = synth.block_inputs(synth.QWEN_Q4, 2)
    b = synth.block_inputs(synth.QWEN_Q4, 2)
    assert torch.equal(a.x, b.x) and torch.equal(a.logits, b.logits)
    assert a.x.dtype == torch.float32 and a.x.shape == (2, 4096)
    assert a.shared_gate_w.dtype == torch.int16
