"""Seeded synthetic inputs for the batch-1 quantised MoE expert block.

This module only draws numbers and packs them into the expert-blob byte
format; it holds none of the block's arithmetic (no dequantisation, no
matrix-vector product, no routing, no activation).  Both the CUDA path and
the fp64 oracle take their inputs from here, so the two never feed each
other.

Two kinds of draws:

* Expert weights (the big part, up to tens of GB) come from a counter-based
  hash.  A word's value depends only on (seed, layer, expert, plane, word
  index), so any single expert can be regenerated alone, on the CPU or on a
  CUDA device, bit-identically: the hash uses only int64 integer operations
  whose products stay below 2**63, and the float steps are single correctly
  rounded fp32 operations followed by a round-to-nearest-even cast to bf16.
* Activations (x, router logits, residual, shared-gate vector) are small and
  are always drawn on the CPU with ``torch.Generator`` and then moved.

Blob format written here (one contiguous blob per expert):

    gate/up rows, r = 0..I-1, each padded to a multiple of 16 bytes:
        gate_q [H*bits/32] uint32   packed codes of gate row r
        up_q   [H*bits/32] uint32   packed codes of up row r
        gate_sb [H/64]     uint32   low half = scale (bf16), high half = bias (bf16)
        up_sb   [H/64]     uint32
    the down projection by column, i = 0..I-1, starting on a 256-byte boundary:
        down_q [H*bits/32] uint32   word w: codes of rows w*(32/bits).. of column i
    its (scale, bias) words by group of 64 columns, g = 0..I/64-1, starting on
    a 256-byte boundary:
        down_sb [H]        uint32   word j: row j's scale and bias for group g
    the blob is padded to a multiple of 256 bytes.

Element c of a packed gate/up row sits at bits (c % (32/bits))*bits of word
c/(32/bits); row j of a down column likewise at bits (j % (32/bits))*bits of
word j/(32/bits).  A range of gate/up rows, a range of down columns and a
range of down groups are each one contiguous byte range.

The packed-code and affine-group form follows the flash-moe write-ups'
description of the 4-bit / 2-bit expert weights ("nibble * scale + bias",
section on the FMA-optimised dequant kernel); the plane order, bit order and
the (scale, bias) pairing are this project's own choice, since the pages do
not fix them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

GROUP = 64
PLANE_ALIGN = 256
PLANES = ("gate_q", "gate_sb", "up_q", "up_sb", "down_q", "down_sb")
_M32 = 0xFFFFFFFF


# ---------------------------------------------------------------------------
# workload shapes
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class BlockShape:
    """Shape and value distributions of one MoE block workload."""

    name: str
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    has_shared: bool
    bits: int
    scale_lo: float
    scale_hi: float
    bias_lo: float
    bias_hi: float
    seed: int
    n_layers: int = 1
    tokens: tuple = (1,)
    zipf_s: Optional[float] = None
    eps: float = 1e-6


# Tiny correctness block: H 512, 8 experts, top-2, no shared expert, I 128, 4-bit.
TINY = BlockShape("tiny_h512_e8_top2_i128_q4", 512, 128, 8, 2, False, 4,
                  0.002, 0.02, -0.1, 0.0, seed=0)
# Qwen-shaped block: H 4096, 512 experts, top-4 + 1 shared expert, I 1024, 4-bit.
QWEN_Q4 = BlockShape("qwen_h4096_e512_top4_shared_i1024_q4", 4096, 1024, 512, 4,
                     True, 4, 0.002, 0.02, -0.1, 0.0, seed=1)
# The same block with 2-bit codes.
QWEN_Q2 = BlockShape("qwen_h4096_e512_top4_shared_i1024_q2", 4096, 1024, 512, 4,
                     True, 2, 0.01, 0.05, -0.1, 0.0, seed=2)
# The 4-bit block at batch 1..16 with Zipf(1.1) expert popularity.
QWEN_Q4_BATCH = BlockShape("qwen_h4096_e512_top4_shared_i1024_q4_zipf", 4096, 1024,
                           512, 4, True, 4, 0.002, 0.02, -0.1, 0.0, seed=3,
                           tokens=(1, 2, 4, 8, 16), zipf_s=1.1)
# 48-layer decode stack: H 2048, 512 experts, top-10, I 512, 4-bit, no shared.
STACK48 = BlockShape("stack48_h2048_e512_top10_i512_q4", 2048, 512, 512, 10, False,
                     4, 0.002, 0.02, -0.1, 0.0, seed=4, n_layers=48, tokens=(256,))

SHAPES = {s.name: s for s in (TINY, QWEN_Q4, QWEN_Q2, QWEN_Q4_BATCH, STACK48)}


# ---------------------------------------------------------------------------
# blob byte format (this module's own copy; the oracle and the C library
# each compute it independently)
# ---------------------------------------------------------------------------
def _round_up(n: int, a: int) -> int:
    return (n + a - 1) // a * a


def plane_words(bits: int, hidden: int, inter: int) -> dict:
    """(rows, words per row) of each of the six parts of a blob; a "row" of
    down_q is a column of the down projection, a row of down_sb a group."""
    per = 32 // bits
    return {
        "gate_q": (inter, hidden // per),
        "gate_sb": (inter, hidden // GROUP),
        "up_q": (inter, hidden // per),
        "up_sb": (inter, hidden // GROUP),
        "down_q": (inter, hidden // per),
        "down_sb": (inter // GROUP, hidden),
    }


def row_layout(bits: int, hidden: int, inter: int) -> tuple:
    """(dict part -> (byte offset of row 0, byte stride between rows), blob bytes)."""
    qh, sh = hidden * bits // 8, hidden // GROUP * 4
    gu_row = _round_up(2 * qh + 2 * sh, 16)
    dq_off = _round_up(inter * gu_row, PLANE_ALIGN)
    dcol = hidden * bits // 8
    dsb_off = _round_up(dq_off + inter * dcol, PLANE_ALIGN)
    parts = {
        "gate_q": (0, gu_row),
        "up_q": (qh, gu_row),
        "gate_sb": (2 * qh, gu_row),
        "up_sb": (2 * qh + sh, gu_row),
        "down_q": (dq_off, dcol),
        "down_sb": (dsb_off, hidden * 4),
    }
    return parts, _round_up(dsb_off + inter // GROUP * hidden * 4, PLANE_ALIGN)


def blob_bytes(bits: int, hidden: int, inter: int) -> int:
    return row_layout(bits, hidden, inter)[1]


# ---------------------------------------------------------------------------
# counter-based hash (int64 tensors holding values in [0, 2**32))
# ---------------------------------------------------------------------------
def _mix32(x: torch.Tensor) -> torch.Tensor:
    # xorshift-multiply finaliser; both odd multipliers are < 2**31 so that
    # (x < 2**32) * c < 2**63 never overflows int64 on any device.
    x = x ^ (x >> 16)
    x = (x * 0x21F0AAAD) & _M32
    x = x ^ (x >> 15)
    x = (x * 0x735A2D97) & _M32
    x = x ^ (x >> 15)
    return x


def _mix32_int(v: int) -> int:
    return int(_mix32(torch.tensor([v & _M32], dtype=torch.int64))[0])


def _stream_key(*parts: int) -> int:
    k = 0x6A09E667
    for p in parts:
        k = _mix32_int(k ^ (p & _M32))
    return k


def _word_hash(key: int, expert: torch.Tensor, index: torch.Tensor) -> torch.Tensor:
    """uint32 (as int64) of word `index` of expert `expert` in stream `key`.

    expert and index broadcast against each other.
    """
    k2 = _mix32_int(key ^ 0x9E3779B9)
    e = _mix32(expert ^ key)
    return _mix32(_mix32(index ^ e) ^ k2)


def _uniform_bf16_bits(h: torch.Tensor, lo: float, hi: float) -> torch.Tensor:
    """bf16 bit patterns (int64 in [0, 65536)) of U(lo, hi) draws from hashes h."""
    device = h.device
    u = (h >> 8).to(torch.float32) * (2.0 ** -24)            # exact, in [0, 1)
    span = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    base = torch.tensor(lo, dtype=torch.float32, device=device)
    v = u * span                                              # one fp32 rounding
    v = v + base                                              # one fp32 rounding
    return v.to(torch.bfloat16).view(torch.int16).to(torch.int64) & 0xFFFF


_PLANE_ID = {name: i for i, name in enumerate(PLANES)}


def expert_blobs(shape: BlockShape, layer: int, experts, device="cpu",
                 seed: Optional[int] = None) -> torch.Tensor:
    """Blobs of the given expert ids as an int32 tensor [n][blob_bytes/4].

    An id >= shape.n_experts denotes a shared expert (id n_experts + j is the
    j-th distinct shared expert); routed and shared experts use the same
    streams, so ids never collide.
    """
    seed = shape.seed if seed is None else seed
    bits, H, I = shape.bits, shape.hidden, shape.inter
    parts, nbytes = row_layout(bits, H, I)
    ex = torch.as_tensor(experts, dtype=torch.int64).reshape(-1, 1).to(device)
    words = torch.zeros((ex.shape[0], nbytes // 4), dtype=torch.int64, device=device)
    for name, (rows, wpr) in plane_words(bits, H, I).items():
        n = rows * wpr
        base, stride = parts[name]
        pid = _PLANE_ID[name]
        idx = torch.arange(n, dtype=torch.int64, device=device)
        dst = base // 4 + (idx // wpr) * (stride // 4) + idx % wpr
        idx = idx.reshape(1, -1)
        if name.endswith("_q"):
            vals = _word_hash(_stream_key(seed, layer, pid, 0), ex, idx)
        else:
            s = _uniform_bf16_bits(_word_hash(_stream_key(seed, layer, pid, 1), ex, idx),
                                   shape.scale_lo, shape.scale_hi)
            b = _uniform_bf16_bits(_word_hash(_stream_key(seed, layer, pid, 2), ex, idx),
                                   shape.bias_lo, shape.bias_hi)
            vals = s | (b << 16)
        words[:, dst] = vals
    # reinterpret the low 32 bits as int32
    return (words - ((words >> 31) << 32)).to(torch.int32)


def expert_blob(shape: BlockShape, layer: int, expert: int, device="cpu",
                seed: Optional[int] = None) -> torch.Tensor:
    """One expert's blob as a flat int32 tensor of blob_bytes/4 words."""
    return expert_blobs(shape, layer, [expert], device, seed)[0]


def fill_pool(out: torch.Tensor, shape: BlockShape, layer: int, first_expert: int,
              count: int, seed: Optional[int] = None, chunk: int = 32) -> None:
    """Write `count` consecutive expert blobs (ids first_expert..) into `out`.

    `out` is a flat int32 tensor (any device) of at least count*blob_bytes/4
    words; generation runs on out's device, `chunk` experts at a time.
    """
    nw = blob_bytes(shape.bits, shape.hidden, shape.inter) // 4
    assert out.dtype == torch.int32 and out.numel() >= count * nw
    view = out[:count * nw].view(count, nw)
    for j in range(0, count, chunk):
        n = min(chunk, count - j)
        ids = list(range(first_expert + j, first_expert + j + n))
        view[j:j + n] = expert_blobs(shape, layer, ids, device=out.device, seed=seed)


# ---------------------------------------------------------------------------
# activations
# ---------------------------------------------------------------------------
def _gen(seed: int, tag: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + tag * 7919) & 0x7FFFFFFFFFFF)
    return g


def normal(seed: int, tag: int, shape_: tuple, std: float = 1.0) -> torch.Tensor:
    """fp32 N(0, std^2) draws on the CPU."""
    t = torch.randn(shape_, generator=_gen(seed, tag), dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t


def shared_gate_vector(shape: BlockShape, layer: int = 0, seed: Optional[int] = None) -> torch.Tensor:
    """bf16 bit patterns (int16 tensor) of w_sg ~ N(0, 1/H)."""
    seed = shape.seed if seed is None else seed
    w = normal(seed, 100 + layer, (shape.hidden,), std=1.0 / math.sqrt(shape.hidden))
    return w.to(torch.bfloat16).view(torch.int16)


def dense_matrix(n_rows: int, hidden: int, bits: int, seed: int, tag: int = 0, scale=(0.002, 0.02),
                 bias=(-0.1, 0.0), device="cpu") -> torch.Tensor:
    """A dense quantised matrix (o_proj) as int32 words: n_rows records of the
    row's codes, then its (scale,bias) words (one per 64 columns), padded to
    16 bytes; codes uniform, scale U(scale), bias U(bias) as bf16."""
    qw, sw = hidden * bits // 32, hidden // GROUP
    rw = _round_up((qw + sw) * 4, 16) // 4
    rows = torch.arange(n_rows, dtype=torch.int64, device=device).reshape(-1, 1)
    words = torch.zeros((n_rows, rw), dtype=torch.int64, device=device)
    words[:, :qw] = _word_hash(_stream_key(seed, tag, 7, 0), rows,
                               torch.arange(qw, dtype=torch.int64, device=device).reshape(1, -1))
    gi = torch.arange(sw, dtype=torch.int64, device=device).reshape(1, -1)
    s = _uniform_bf16_bits(_word_hash(_stream_key(seed, tag, 7, 1), rows, gi), scale[0], scale[1])
    b = _uniform_bf16_bits(_word_hash(_stream_key(seed, tag, 7, 2), rows, gi), bias[0], bias[1])
    words[:, qw:qw + sw] = s | (b << 16)
    return (words - ((words >> 31) << 32)).to(torch.int32).reshape(-1)


def norm_weight(hidden: int, seed: int, tag: int = 0) -> torch.Tensor:
    """A learned RMSNorm weight stand-in: fp32 1 + N(0, 0.1^2)."""
    return 1.0 + normal(seed, 200 + tag, (hidden,), std=0.1)


def router_matrix(shape: BlockShape, layer: int = 0, seed: Optional[int] = None) -> torch.Tensor:
    """bf16 bit patterns (int16 tensor [E][H]) of W_r ~ N(0, 1/H): with x ~ N(0, 1)
    the logits are about N(0, 1), as the workloads' router logits."""
    seed = shape.seed if seed is None else seed
    w = normal(seed, 300 + layer, (shape.n_experts, shape.hidden), std=1.0 / math.sqrt(shape.hidden))
    return w.to(torch.bfloat16).view(torch.int16)


def zipf_logits(seed: int, tag: int, n_tokens: int, n_experts: int, s: float) -> torch.Tensor:
    """Router logits whose top-K is a Plackett-Luce draw from Zipf(s) popularity.

    logit_e = log p_e + Gumbel(0,1), p_e proportional to (rank_e + 1)^-s with a
    seeded random rank permutation shared by all tokens.
    """
    g = _gen(seed, tag)
    rank = torch.randperm(n_experts, generator=g)
    logp = -s * torch.log((rank + 1).to(torch.float64))
    u = torch.rand((n_tokens, n_experts), generator=g, dtype=torch.float64)
    u = u.clamp(1e-300, 1.0 - 1e-16)
    gumbel = -torch.log(-torch.log(u))
    return (logp.unsqueeze(0) + gumbel).to(torch.float32)


@dataclass
class BlockInputs:
    """Activations of one call: x [T][H], logits [T][E], residual [T][H]."""

    x: torch.Tensor
    logits: torch.Tensor
    residual: torch.Tensor
    shared_gate_w: Optional[torch.Tensor] = None  # int16 bf16 bits [H]


def block_inputs(shape: BlockShape, n_tokens: int = 1, tag: int = 0,
                 seed: Optional[int] = None) -> BlockInputs:
    seed = shape.seed if seed is None else seed
    H, E = shape.hidden, shape.n_experts
    x = normal(seed, 10 + 4 * tag, (n_tokens, H))
    if shape.zipf_s is not None:
        logits = zipf_logits(seed, 11 + 4 * tag, n_tokens, E, shape.zipf_s)
    else:
        logits = normal(seed, 11 + 4 * tag, (n_tokens, E))
    residual = normal(seed, 12 + 4 * tag, (n_tokens, H))
    wsg = shared_gate_vector(shape, 0, seed) if shape.has_shared else None
    return BlockInputs(x, logits, residual, wsg)


def stack_inputs(shape: BlockShape, n_tokens: int, tag: int = 0,
                 seed: Optional[int] = None) -> tuple:
    """(h0 [T][H], logits [T][L][E]) for independent decode tokens."""
    seed = shape.seed if seed is None else seed
    h0 = normal(seed, 50 + 2 * tag, (n_tokens, shape.hidden))
    logits = normal(seed, 51 + 2 * tag, (n_tokens, shape.n_layers, shape.n_experts))
    return h0, logits
