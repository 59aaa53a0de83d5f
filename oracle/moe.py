"""Plain fp64 definitions of the quantised MoE expert block (test oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the product library.

Sources (page title, then section):
  [FM]  "flash-moe: C/Metal engine running a 397B MoE on an M3 Max"
        (discuss.pytorch.kr): sections "FMA-optimised dequant kernel",
        "hand-written Metal compute shaders", "per-layer pipeline",
        "Qwen3.5-397B-A17B model architecture".
  [GN]  "Flash-MoE - running a 397B-parameter model on a laptop" (GeekNews
        topic 27758), sections "Model architecture", "Metal Compute Shaders".
"""
from __future__ import annotations

import numpy as np

GROUP = 64          # quantisation group: 64 consecutive input columns of a row
_ALIGN = 256        # the down parts and the blob size are aligned to 256 bytes


# ---------------------------------------------------------------------------
# packed expert blob
# ---------------------------------------------------------------------------
def layout(bits: int, hidden: int, inter: int) -> tuple:
    """Where the six parts of an expert blob live.

    Gate/up row r (r < I) is one record of gate codes, up codes, gate
    (scale,bias) words and up (scale,bias) words, padded to a multiple of 16
    bytes.  The down projection follows from the next 256-byte boundary,
    stored by column: column i (i < I) is H*bits/8 bytes whose word w holds
    the codes of rows w*(32/bits) .. (w+1)*(32/bits)-1 of that column.  Its
    (scale,bias) words follow from the next 256-byte boundary, by group:
    group g (columns 64g .. 64g+63) is H words, word j for row j.  The blob
    is padded to a multiple of 256 bytes.  Returns
    (dict name -> (offset of row 0, row stride, rows, 32-bit words per row),
    blob_bytes), all in bytes except the word count; for the two down parts
    a "row" is a column (down_q) or a group (down_sb).
    Pinned by the expert-size pin (6.75 MiB per 4-bit expert of the
    397B model, [FM] "SSD expert streaming") and by blobs built field by
    field from chosen codes.
    """
    if bits not in (2, 4):
        raise ValueError("bits must be 2 or 4")
    per_word = 32 // bits
    qh, sh = hidden // per_word * 4, hidden // GROUP * 4       # bytes of one gate/up row's parts
    gu_stride = -(-(2 * qh + 2 * sh) // 16) * 16
    dq_base = -(-(inter * gu_stride) // _ALIGN) * _ALIGN
    dcol = hidden // per_word * 4                              # bytes of one down column
    dsb_base = -(-(dq_base + inter * dcol) // _ALIGN) * _ALIGN
    out = {
        "gate_q": (0, gu_stride, inter, qh // 4),
        "up_q": (qh, gu_stride, inter, qh // 4),
        "gate_sb": (2 * qh, gu_stride, inter, sh // 4),
        "up_sb": (2 * qh + sh, gu_stride, inter, sh // 4),
        "down_q": (dq_base, dcol, inter, hidden // per_word),
        "down_sb": (dsb_base, hidden * 4, inter // GROUP, hidden),
    }
    return out, -(-(dsb_base + inter // GROUP * hidden * 4) // _ALIGN) * _ALIGN


def unpack_codes(words: np.ndarray, bits: int) -> np.ndarray:
    """Integer codes of packed rows: uint32 [rows][wpr] -> int64 [rows][wpr*32/bits].

    Code c sits at bit (c mod (32/bits))*bits of word c div (32/bits), lowest
    bits first.  Pinned by hand-worked words (tests/golden/unpack_examples.txt).
    """
    w = np.asarray(words, dtype=np.uint64)
    per_word = 32 // bits
    mask = (1 << bits) - 1
    codes = np.empty(w.shape[:-1] + (w.shape[-1], per_word), dtype=np.int64)
    for i in range(per_word):
        codes[..., i] = ((w >> np.uint64(bits * i)) & np.uint64(mask)).astype(np.int64)
    return codes.reshape(w.shape[:-1] + (w.shape[-1] * per_word,))


def bf16_to_f64(b16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values (bf16 is the top half of fp32)."""
    u = (np.asarray(b16, dtype=np.uint32) & 0xFFFF) << 16
    return u.view(np.float32).astype(np.float64)


def dequantize(q_words: np.ndarray, sb_words: np.ndarray, bits: int) -> np.ndarray:
    """W[r, c] = q[r, c] * s[r, c//64] + b[r, c//64] in fp64, from packed rows.

    [FM] "FMA-optimised dequant kernel": the weight is nibble*scale+bias.
    sb word g of a row holds scale (low 16 bits, bf16) and bias (high 16).
    Pinned by hand-worked dequant examples and the FMA identity.
    """
    return dequantize_codes(unpack_codes(q_words, bits), sb_words)


def dequantize_codes(q: np.ndarray, sb_words: np.ndarray) -> np.ndarray:
    """W[r, c] = q[r, c] * s[r, c//64] + b[r, c//64] from integer codes q [rows][n]
    and (scale,bias) words [rows][n/64]."""
    q = np.asarray(q).astype(np.float64)
    sb = np.asarray(sb_words, dtype=np.uint32)
    s = bf16_to_f64(sb & 0xFFFF)
    b = bf16_to_f64(sb >> 16)
    n = q.shape[-1]
    if n != sb.shape[-1] * GROUP:
        raise ValueError("codes and (scale,bias) groups disagree")
    g = np.arange(n) // GROUP
    return q * s[..., g] + b[..., g]


def part_rows(blob: np.ndarray, bits: int, hidden: int, inter: int, name: str, n=None) -> np.ndarray:
    """The first n (default: all) rows of one part of a blob, uint32 [n][words per row]."""
    words = np.ascontiguousarray(blob).view(np.uint32).reshape(-1)
    parts, nbytes = layout(bits, hidden, inter)
    if words.size * 4 < nbytes:
        raise ValueError("blob too small")
    off, stride, rows, wpr = parts[name]
    n = rows if n is None else n
    index = (off + np.arange(n)[:, None] * stride) // 4 + np.arange(wpr)[None, :]
    return words[index]


def expert_weights(blob: np.ndarray, bits: int, hidden: int, inter: int) -> tuple:
    """(Wg [I][H], Wu [I][H], Wd [H][I]) dequantised from one blob (fp64).

    The down codes are stored by column and its (scale,bias) words by group
    (see layout); both are turned to row-major [H][...] before the same
    dequantisation as the gate and up rows.
    """

    def plane(name):
        return part_rows(blob, bits, hidden, inter, name)

    wg = dequantize(plane("gate_q"), plane("gate_sb"), bits)
    wu = dequantize(plane("up_q"), plane("up_sb"), bits)
    wd = dequantize_codes(unpack_codes(plane("down_q"), bits).T, plane("down_sb").T)
    return wg, wu, wd


# ---------------------------------------------------------------------------
# expert FFN
# ---------------------------------------------------------------------------
def silu(a):
    """a * sigmoid(a) = a / (1 + exp(-a))."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def expert_ffn(weights: tuple, x: np.ndarray) -> np.ndarray:
    """y = Wd (silu(Wg x) * (Wu x)).

    [FM] shader list: dequant matvec for gate/up/down and fused SwiGLU
    (gate branch through SiLU, multiplied by the up branch).
    Pinned by the constant-row closed form.
    """
    wg, wu, wd = weights
    x = np.asarray(x, dtype=np.float64)
    a = wg @ x
    u = wu @ x
    h = silu(a) * u
    return wd @ h


# ---------------------------------------------------------------------------
# routing, shared gate, combine
# ---------------------------------------------------------------------------
def route(logits: np.ndarray, k: int) -> tuple:
    """(ids [K] int, weights [K] fp64) for one token.

    [FM] "per-layer pipeline": softmax + top-K on the router logits.  The K
    largest logits are taken by value, ties broken towards the lower expert
    id, in descending order; the weights are the softmax of the K selected
    logits (equal to full softmax -> top-K -> renormalise).
    Pinned by brute force over all K-subsets and the sum-to-one invariant.
    """
    l = np.asarray(logits, dtype=np.float64)
    if not np.all(np.isfinite(l)):
        raise ValueError("router logits must be finite")
    if not 1 <= k <= l.size:
        raise ValueError("need 1 <= K <= number of experts")
    order = np.argsort(-l, kind="stable")       # stable: equal logits keep id order
    ids = order[:k]
    sel = l[ids]
    e = np.exp(sel - sel.max())
    return ids.astype(np.int64), e / e.sum()


def shared_gate(wsg_bf16: np.ndarray, x: np.ndarray) -> float:
    """g = sigmoid(w_sg . x) with w_sg given as bf16 bit patterns.

    [FM] shader list "MoE combine + residual + sigmoid gate" and model
    section "plus one shared expert".  Pinned by closed-form gate values.
    """
    w = bf16_to_f64(wsg_bf16)
    return float(sigmoid(w @ np.asarray(x, dtype=np.float64)))


def dense_record_words(bits: int, hidden: int) -> tuple:
    """A dense quantised matrix (o_proj) is N row records, each the row's
    codes (hidden*bits/32 words, lowest bits first) then its (scale,bias)
    words (one per 64 columns), padded to a multiple of 16 bytes.  Returns
    (code words, scale words, words per record)."""
    qw = hidden * bits // 32
    sw = hidden // GROUP
    return qw, sw, -(-(qw + sw) * 4 // 16) * 16 // 4


def dense_weights(words: np.ndarray, bits: int, n_rows: int, hidden: int) -> np.ndarray:
    """W [N][H] fp64 of a dense quantised matrix given as uint32 words.
    Pinned by records built field by field from random codes and dyadic
    scales/biases, read back exactly."""
    qw, sw, rw = dense_record_words(bits, hidden)
    rec = np.asarray(words, dtype=np.uint32).reshape(n_rows, rw)
    return dequantize(rec[:, :qw], rec[:, qw:qw + sw], bits)


def dense_matvec(w: np.ndarray, x: np.ndarray, residual=None) -> np.ndarray:
    """y = W x (+ residual) for one token [H] or T tokens [T][H]: the o_proj
    of [FM] "per-layer pipeline" (CMD2), a dense 4-bit matvec."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
    return y if residual is None else y + np.asarray(residual, dtype=np.float64)


def router_logits(w_router_bf16: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Router logits l = W_r x of one token (x [H] -> [E]) or of T tokens
    (x [T][H] -> [T][E]), W_r [E][H] given as bf16 bit patterns.

    [FM] "per-layer pipeline": the second command buffer computes the routing
    logits on the GPU (with o_proj, the norm and the shared expert) before the
    CPU's softmax + top-K.  The pages give no storage type for W_r; bf16 is
    this project's reading, as for w_sg.  Pinned by hand-worked values, exact
    integer products checked against Python integers, and one-hot rows.
    """
    w = bf16_to_f64(w_router_bf16)
    return np.asarray(x, dtype=np.float64) @ w.T


def combine(residual, routed_y, weights, shared_y=None, g=None):
    """out = residual + sum_k w_k y_k (+ g * y_shared)."""
    out = np.asarray(residual, dtype=np.float64).copy()
    for wk, yk in zip(weights, routed_y):
        out += wk * yk
    if shared_y is not None:
        out += g * shared_y
    return out


def moe_block(get_expert, x, logits, residual, k, shared=None, wsg=None):
    """One MoE block for T independent tokens.

    get_expert(e) -> (Wg, Wu, Wd) of routed expert e;  shared -> the shared
    expert's weights or None.  x, residual: [T][H]; logits: [T][E].
    Returns dict(out [T][H], ids [T][K], weights [T][K], gate [T] or None,
    y [T][K(+1)][H] unweighted expert outputs).
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    residual = np.atleast_2d(np.asarray(residual, dtype=np.float64))
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    T = x.shape[0]
    cache = {}
    outs, all_ids, all_w, gates, ys = [], [], [], [], []
    for t in range(T):
        ids, w = route(logits[t], k)
        y_t = []
        for e in ids:
            e = int(e)
            if e not in cache:
                cache[e] = get_expert(e)
            y_t.append(expert_ffn(cache[e], x[t]))
        ysh, g = None, None
        if shared is not None:
            ysh = expert_ffn(shared, x[t])
            g = shared_gate(wsg, x[t])
        outs.append(combine(residual[t], y_t, w, ysh, g))
        all_ids.append(ids)
        all_w.append(w)
        gates.append(g)
        ys.append(np.stack(y_t + ([ysh] if ysh is not None else [])))
    return {
        "out": np.stack(outs),
        "ids": np.stack(all_ids),
        "weights": np.stack(all_w),
        "gate": None if shared is None else np.array(gates),
        "y": np.stack(ys),
    }


# ---------------------------------------------------------------------------
# stacked decode
# ---------------------------------------------------------------------------
def rms_norm(h, eps: float, weight=None):
    """h / sqrt(mean(h^2) + eps), times a learned weight vector when one is
    given ([FM] shader list: RMSNorm; "per-layer pipeline": the norm of CMD2).
    Pinned by constant vectors, unit-weight identity and linearity in the
    weight."""
    h = np.asarray(h, dtype=np.float64)
    x = h / np.sqrt(np.mean(h * h) + eps)
    return x if weight is None else x * np.asarray(weight, dtype=np.float64)


def stack_decode(get_expert_l, h0, logits, k, eps, shared_l=None, wsg_l=None):
    """One token through L pre-norm MoE blocks.

    h_{l+1} = h_l + MoE_l(rms_norm(h_l)), the residual being h_l itself
    ([FM] "deferred CMD3": combine, residual and norm stay on the GPU and
    feed the next layer).  get_expert_l(l, e) -> weights of expert e of layer
    l; logits [L][E].  Returns (h_L, ids [L][K]).
    """
    h = np.asarray(h0, dtype=np.float64).copy()
    logits = np.asarray(logits, dtype=np.float64)
    all_ids = []
    for l in range(logits.shape[0]):
        xn = rms_norm(h, eps)
        sh = None if shared_l is None else shared_l(l)
        wsg = None if wsg_l is None else wsg_l(l)
        r = moe_block(lambda e, l=l: get_expert_l(l, e), xn[None], logits[l][None],
                      h[None], k, sh, wsg)
        h = r["out"][0]
        all_ids.append(r["ids"][0])
    return h, np.stack(all_ids)
