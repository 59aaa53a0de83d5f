"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``pin_*`` function checks the oracle against one of:
  * hand-worked values stored in tests/golden/ (each file cites its page);
  * the flash-moe write-up's own identity (nibble*scale+bias)*x ==
    fma(nibble, scale*x, bias*x), evaluated exactly with fractions;
  * closed forms (constant-code experts, designed logits, constant vectors);
  * brute force over all K-subsets for the top-K;
  * invariants (weights sum to one, zero-weight experts change nothing);
  * sizes printed on the pages (6.75 MB per expert, 209 GB vs 120 GB).

``test_planted_mistakes`` plants plausible mistakes in the oracle (on the
CPU) and checks that at least one pin catches each of them.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle.moe as om
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# test-side helpers: packing codes and building blobs from chosen values
# ---------------------------------------------------------------------------
def pack(codes, bits):
    """Pack integer codes [rows][n] into uint32 words, code c at bits*(c mod 32/bits)."""
    c = np.asarray(codes, dtype=np.uint64)
    per = 32 // bits
    rows, n = c.shape
    c = c.reshape(rows, n // per, per)
    w = np.zeros((rows, n // per), dtype=np.uint64)
    for i in range(per):
        w |= c[..., i] << np.uint64(bits * i)
    return w.astype(np.uint32)


def bf16(v):
    """bf16 bit pattern of a value that bf16 represents exactly."""
    b = np.float32(v).view(np.uint32)
    assert b & 0xFFFF == 0, f"{v} is not exactly representable in bf16"
    return int(b >> 16)


def sb(scale, bias, rows, groups):
    return np.full((rows, groups), bf16(scale) | (bf16(bias) << 16), dtype=np.uint32)


def _up(n, a):
    return -(-n // a) * a


def build_blob(bits, H, I, gate, up, down):
    """Blob bytes from (codes, sb_words) per matrix, written field by field.

    The test's own statement of the packed format: I gate/up records of
    [gate codes | up codes | gate (scale,bias) words | up words], each padded
    to 16 bytes; from the next 256-byte boundary the down projection by
    column (column i: H codes packed over rows, lowest bits first); from the
    next 256-byte boundary the down (scale,bias) words by group of 64 columns
    (group g: one word per row); the blob padded to 256 bytes.  Codes are
    [rows][cols] of the matrix as used (gate/up [I][H], down [H][I]).
    """
    per = 32 // bits
    qh, sh = H // per * 4, H // 64 * 4
    gu = _up(2 * qh + 2 * sh, 16)
    dq = _up(I * gu, 256)
    dcol = H // per * 4
    dsb = _up(dq + I * dcol, 256)
    nbytes = _up(dsb + I // 64 * H * 4, 256)
    words = np.zeros(nbytes // 4, dtype=np.uint32)

    def put(byte_off, vals):
        vals = np.asarray(vals, dtype=np.uint32)
        words[byte_off // 4: byte_off // 4 + vals.size] = vals

    gq, gsb = pack(gate[0], bits), np.asarray(gate[1], dtype=np.uint32)
    uq, usb = pack(up[0], bits), np.asarray(up[1], dtype=np.uint32)
    for r in range(gq.shape[0]):
        put(r * gu, gq[r])
        put(r * gu + qh, uq[r])
        put(r * gu + 2 * qh, gsb[r])
        put(r * gu + 2 * qh + sh, usb[r])
    dcodes = np.asarray(down[0])                      # [H][I]
    dcols = pack(dcodes.T, bits)                      # [I][H/per]: column i packed over rows
    dsbw = np.asarray(down[1], dtype=np.uint32)       # [H][I/64]
    for i in range(dcols.shape[0]):
        put(dq + i * dcol, dcols[i])
    for g in range(dsbw.shape[1]):
        put(dsb + g * H * 4, dsbw[:, g])
    return words.view(np.uint8)


def const_expert(bits, H, I, cg, sg, bg, cu, su, bu, cd, sd, bd):
    full = lambda rows, n, c: np.full((rows, n), c, dtype=np.int64)
    return build_blob(
        bits, H, I,
        (full(I, H, cg), sb(sg, bg, I, H // 64)),
        (full(I, H, cu), sb(su, bu, I, H // 64)),
        (full(H, I, cd), sb(sd, bd, H, I // 64)),
    )


def const_ffn(H, I, X, cg, sg, bg, cu, su, bu, cd, sd, bd):
    """Closed form of y for a constant-code expert and sum(x) = X."""
    a = (cg * sg + bg) * X
    u = (cu * su + bu) * X
    h = a / (1.0 + math.exp(-a)) * u
    return (cd * sd + bd) * I * h


def read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------
def pin_unpack_golden():
    for row in read_rows("unpack_examples.txt"):
        bits, word, codes = int(row[0]), int(row[1], 16), [int(v) for v in row[2:]]
        got = om.unpack_codes(np.array([[word]], dtype=np.uint32), bits)[0]
        assert list(got) == codes, (bits, hex(word), list(got), codes)


def pin_dequant_golden():
    for row in read_rows("dequant_examples.txt"):
        bits, q = int(row[0]), int(row[1])
        s16, b16, want = int(row[2], 16), int(row[3], 16), float(row[4])
        codes = np.full((1, 64), q, dtype=np.int64)
        sbw = np.array([[s16 | (b16 << 16)]], dtype=np.uint32)
        w = om.dequantize(pack(codes, bits), sbw, bits)
        assert w.shape == (1, 64)
        assert np.all(w == want), (row, w[0, :4])


def pin_two_groups():
    # group 0: scale 1, bias 0 -> w = q;  group 1: scale 0, bias 5 -> w = 5
    codes = (np.arange(128) % 16).reshape(1, 128)
    sbw = np.array([[bf16(1.0) | (bf16(0.0) << 16), bf16(0.0) | (bf16(5.0) << 16)]],
                   dtype=np.uint32)
    w = om.dequantize(pack(codes, 4), sbw, 4)[0]
    assert np.array_equal(w[:64], codes[0, :64].astype(np.float64))
    assert np.all(w[64:] == 5.0)


def _dyadic_case(bits, rng, H=128, I=64):
    """A small expert whose values are all short dyadic rationals."""
    cmax = (1 << bits) - 1
    scales = [2.0 ** -6, 3 * 2.0 ** -7, 2.0 ** -5, 5 * 2.0 ** -8]
    biases = [-(2.0 ** -4), -(3 * 2.0 ** -6), 0.0, -(2.0 ** -3)]

    def mat(rows, n):
        codes = rng.integers(0, cmax + 1, size=(rows, n))
        sbw = np.zeros((rows, n // 64), dtype=np.uint32)
        sv = np.zeros((rows, n // 64))
        bv = np.zeros((rows, n // 64))
        for r in range(rows):
            for g in range(n // 64):
                s, b = scales[rng.integers(4)], biases[rng.integers(4)]
                sbw[r, g] = bf16(s) | (bf16(b) << 16)
                sv[r, g], bv[r, g] = s, b
        return codes, sbw, sv, bv

    gate, up, down = mat(I, H), mat(I, H), mat(H, I)
    x = rng.integers(-16, 17, size=H) / 8.0
    blob = build_blob(bits, H, I, gate[:2], up[:2], down[:2])
    return blob, gate, x


def pin_fma_identity():
    """Oracle gate matvec == sum_c fma(q_c, s*x_c, b*x_c), exact (fractions)."""
    rng = np.random.default_rng(7)
    for bits in (4, 2):
        H, I = 128, 64
        blob, (codes, _, sv, bv), x = _dyadic_case(bits, rng, H, I)
        wg, _, _ = om.expert_weights(blob, bits, H, I)
        got = wg @ x
        for r in range(I):
            acc = Fraction(0)
            for c in range(H):
                s, b, xc = Fraction(sv[r, c // 64]), Fraction(bv[r, c // 64]), Fraction(x[c])
                acc += int(codes[r, c]) * (s * xc) + b * xc     # fma(q, s*x, b*x)
            assert Fraction(got[r]) == acc, (bits, r)


def pin_group_decomposition():
    """sum_c (q s + b) x == sum_g (s_g sum q x + b_g sum x), exact on dyadic values."""
    rng = np.random.default_rng(11)
    for bits in (4, 2):
        H, I = 128, 64
        blob, (codes, _, sv, bv), x = _dyadic_case(bits, rng, H, I)
        wg, _, _ = om.expert_weights(blob, bits, H, I)
        got = wg @ x
        for r in range(I):
            tot = 0.0
            for g in range(H // 64):
                sl = slice(64 * g, 64 * g + 64)
                tot += sv[r, g] * float(codes[r, sl] @ x[sl]) + bv[r, g] * float(x[sl].sum())
            assert got[r] == tot, (bits, r)


def pin_random_blob_fields():
    """Every code and (scale,bias) word of all three matrices lands where the
    format puts it: random codes and per-(row, group) dyadic scales and
    biases, written field by field, dequantise exactly to q*s+b (a row
    permutation, a stride slip or a transposed plane changes some value)."""
    rng = np.random.default_rng(13)
    scales = [2.0 ** -6, 3 * 2.0 ** -7, 2.0 ** -5, 5 * 2.0 ** -8, 2.0 ** -4]
    biases = [-(2.0 ** -4), -(3 * 2.0 ** -6), 0.0, -(2.0 ** -3), 2.0 ** -7]
    for bits, H, I in ((4, 128, 128), (2, 128, 128), (4, 192, 64), (2, 64, 192)):
        cmax = (1 << bits) - 1

        def mat(rows, n):
            codes = rng.integers(0, cmax + 1, size=(rows, n))
            si = rng.integers(len(scales), size=(rows, n // 64))
            bi = rng.integers(len(biases), size=(rows, n // 64))
            sbw = np.vectorize(lambda a, b: bf16(scales[a]) | (bf16(biases[b]) << 16),
                               otypes=[np.uint32])(si, bi)
            g = np.arange(n) // 64
            want = codes * np.array(scales)[si][:, g] + np.array(biases)[bi][:, g]
            return (codes, sbw), want

        gate, wg = mat(I, H)
        up, wu = mat(I, H)
        down, wd = mat(H, I)
        blob = build_blob(bits, H, I, gate, up, down)
        got = om.expert_weights(blob, bits, H, I)
        for name, g_, w_ in zip(("gate", "up", "down"), got, (wg, wu, wd)):
            assert g_.shape == w_.shape and np.array_equal(g_, w_), (bits, H, I, name)


CONST = dict(cg=3, sg=2.0 ** -6, bg=-(2.0 ** -5),   # gate weight 1/64
             cu=10, su=2.0 ** -6, bu=0.0,            # up weight 10/64
             cd=5, sd=2.0 ** -7, bd=-(2.0 ** -6))    # down weight 3/128


def pin_constant_rows():
    for bits in (4, 2):
        H, I = 128, 64
        c = dict(CONST)
        if bits == 2:
            c.update(cu=2, su=2.0 ** -5, cd=3, sd=2.0 ** -6)
        blob = const_expert(bits, H, I, **c)
        w = om.expert_weights(blob, bits, H, I)
        for x in (np.full(H, 0.25), np.linspace(-1, 2, H), -np.ones(H)):
            y = om.expert_ffn(w, x)
            want = const_ffn(H, I, float(x.sum()), **c)
            assert y.shape == (H,)
            assert np.allclose(y, want, rtol=1e-12, atol=0), (bits, y[:2], want)


def brute_topk(logits, k):
    best_sum, best = None, None
    for sub in itertools.combinations(range(len(logits)), k):   # lexicographic order
        s = sum(logits[i] for i in sub)
        if best_sum is None or s > best_sum:
            best_sum, best = s, sub
    return sorted(best, key=lambda i: (-logits[i], i))


def pin_route_bruteforce():
    rng = np.random.default_rng(3)
    for E in range(1, 11):
        for k in range(1, E + 1):
            for trial in range(4):
                if trial < 2:
                    l = rng.integers(-2, 3, size=E).astype(np.float32)   # many ties
                else:
                    l = rng.standard_normal(E).astype(np.float32)
                if trial == 3 and E > 1:
                    l[0], l[E - 1] = np.float32(-0.0), np.float32(0.0)   # -0 == +0
                    l[1:E - 1] = -1.0
                ids, _ = om.route(l, k)
                assert list(ids) == brute_topk([float(v) for v in l], k), (E, k, l, ids)


def pin_route_weights():
    rng = np.random.default_rng(5)
    for k in (1, 2, 4, 10):
        l = rng.standard_normal(512).astype(np.float32)
        ids, w = om.route(l, k)
        assert abs(w.sum() - 1.0) <= 1e-15
        assert np.all(np.diff(w) <= 0)
        if k == 1:
            assert w[0] == 1.0
    # softmax over the selected logits: log 1, log 2, log 3, log 6 -> 1:2:3:6
    l = np.log(np.array([1.0, 3.0, 2.0, 6.0, 0.5]))
    ids, w = om.route(l, 3)
    assert list(ids) == [3, 1, 2]
    assert np.allclose(w, [6 / 11, 3 / 11, 2 / 11], rtol=1e-14)


def pin_special_values():
    assert om.silu(0.0) == 0.0
    assert om.sigmoid(0.0) == 0.5
    assert abs(om.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert abs(om.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    wsg = np.full(64, bf16(0.125), dtype=np.uint16)
    assert abs(om.shared_gate(wsg, np.full(64, 0.25)) - 1 / (1 + math.exp(-2.0))) < 1e-15
    assert om.shared_gate(np.full(64, bf16(-256.0), dtype=np.uint16), np.ones(64)) == 0.0
    eps = 1e-6
    for c in (3.0, -0.5, 1e-3):
        v = om.rms_norm(np.full(32, c), eps)
        want = math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c))
        assert np.allclose(v, want, rtol=1e-14), (c, v[0], want)


def pin_zero_weight():
    H, I, bits = 128, 64, 4
    rng = np.random.default_rng(2)
    blobs = [synth.expert_blob(synth.TINY, 0, e).numpy().view(np.uint8) for e in range(3)]
    blobs = [om.expert_weights(b, bits, 512, 128) for b in blobs]
    x = rng.standard_normal(512)
    res = rng.standard_normal(512)
    # expert 2's logit is 1e4 below the maximum: its weight underflows to 0
    logits = np.array([1.0, 0.5, 1.0 - 1e4])
    r1 = om.moe_block(lambda e: blobs[e], x, logits, res, 3)
    assert r1["weights"][0][2] == 0.0
    perturbed = list(blobs)
    perturbed[2] = tuple(w * 7.0 + 1.0 for w in blobs[2])
    r2 = om.moe_block(lambda e: perturbed[e], x, logits, res, 3)
    assert np.array_equal(r1["out"], r2["out"])
    # an expert whose scales and biases are all zero contributes nothing
    zero = const_expert(bits, H, I, 5, 0.0, 0.0, 5, 0.0, 0.0, 5, 0.0, 0.0)
    y = om.expert_ffn(om.expert_weights(zero, bits, H, I), rng.standard_normal(H))
    assert np.all(y == 0.0)


def pin_page_sizes():
    facts = {r[0]: float(r[1]) for r in read_rows("page_facts.txt")}
    H = int(facts["hidden"])
    # expert FFN intermediate 1024 makes 3*H*I weights at 4 bits plus one bf16
    # scale and bias per 64 weights: exactly 6.75 MiB, the pages' "6.75MB".
    _, b4 = om.layout(4, H, 1024)
    _, b2 = om.layout(2, H, 1024)
    assert b4 == facts["expert_mb_4bit"] * 2 ** 20
    assert b2 == 3.75 * 2 ** 20
    # 4-bit minus 2-bit totals: the non-expert weights cancel.
    per_model = facts["layers"] * (facts["experts"] + facts["shared"])
    diff_gib = per_model * (b4 - b2) / 2 ** 30
    printed = facts["total_gb_4bit"] - facts["total_gb_2bit"]
    assert abs(diff_gib - printed) / printed < 0.02, (diff_gib, printed)
    # both totals exceed the expert bytes alone by a few GB of dense weights
    for bits, key in ((4, "total_gb_4bit"), (2, "total_gb_2bit")):
        _, b = om.layout(bits, H, 1024)
        extra = facts[key] - per_model * b / 2 ** 30
        assert 0 < extra < 10, (bits, extra)


def pin_layout_matches_generator():
    for bits, H, I in ((4, 512, 128), (4, 4096, 1024), (2, 4096, 1024), (4, 2048, 512), (2, 192, 320)):
        parts, nbytes = om.layout(bits, H, I)
        offs, nb2 = synth.row_layout(bits, H, I)
        assert nbytes == nb2
        assert {k: (v[0], v[1]) for k, v in parts.items()} == offs


def pin_block_closed_form():
    H, I, bits = 64, 64, 4
    consts = [dict(CONST, cg=cg, cd=cd) for cg, cd in ((3, 5), (4, 6), (5, 7), (6, 9))]
    experts = [om.expert_weights(const_expert(bits, H, I, **c), bits, H, I) for c in consts]
    shared_c = dict(CONST, cg=4, cu=12, cd=4)
    shared = om.expert_weights(const_expert(bits, H, I, **shared_c), bits, H, I)
    x = np.full(H, 0.25)                       # sum 16
    wsg = np.full(H, bf16(0.125), dtype=np.uint16)   # w_sg . x = 2
    logits = np.log(np.array([1.0, 3.0, 2.0, 6.0]))
    res = np.linspace(-3, 3, H)
    r = om.moe_block(lambda e: experts[e], x, logits, res, 2, shared, wsg)
    assert list(r["ids"][0]) == [3, 1]
    assert np.allclose(r["weights"][0], [2 / 3, 1 / 3], rtol=1e-14)
    g = 1 / (1 + math.exp(-2.0))
    assert abs(r["gate"][0] - g) < 1e-15
    y3 = const_ffn(H, I, 16.0, **consts[3])
    y1 = const_ffn(H, I, 16.0, **consts[1])
    ys = const_ffn(H, I, 16.0, **shared_c)
    want = res + 2 / 3 * y3 + 1 / 3 * y1 + g * ys
    assert np.allclose(r["out"][0], want, rtol=1e-12, atol=1e-12)


def pin_stack_closed_form():
    H, I, bits, eps = 64, 64, 4, 1e-6
    c0 = dict(CONST)
    c1 = dict(CONST, cg=7, cd=2, bd=2.0 ** -6)
    layers = [[om.expert_weights(const_expert(bits, H, I, **c), bits, H, I) for c in (c0, c1)],
              [om.expert_weights(const_expert(bits, H, I, **c), bits, H, I) for c in (c1, c0)]]
    h0 = np.full(H, 0.75)
    logits = np.array([[0.0, 1.0], [0.5, -0.5]])     # K=1: layer 0 -> expert 1, layer 1 -> expert 0
    h, ids = om.stack_decode(lambda l, e: layers[l][e], h0, logits, 1, eps)
    assert ids.tolist() == [[1], [0]]
    hv = 0.75
    for c in (c1, c1):          # layer 0 expert 1 = c1, layer 1 expert 0 = c1
        xv = hv / math.sqrt(hv * hv + eps)
        hv = hv + const_ffn(H, I, H * xv, **c)
    assert np.allclose(h, hv, rtol=1e-12), (h[0], hv)


def pin_router_logits():
    # hand-worked: rows (1, -2, 0.5, 3), (0, 0, 0, 0.25), (-1, -1, -1, -1) against x = (1, 2, 3, 4)
    W = np.array([[bf16(v) for v in row] for row in ((1, -2, 0.5, 3), (0, 0, 0, 0.25), (-1, -1, -1, -1))],
                 dtype=np.uint16)
    assert list(om.router_logits(W, np.array([1.0, 2.0, 3.0, 4.0]))) == [10.5, 1.0, -10.0]
    rng = np.random.default_rng(11)
    # one-hot rows pick x[perm[e]]: a row shift or a transposed operand fails
    E, H = 7, 96
    perm = rng.permutation(H)[:E]
    onehot = np.zeros((E, H), dtype=np.uint16)
    onehot[np.arange(E), perm] = bf16(1.0)
    x = rng.standard_normal(H)
    assert np.array_equal(om.router_logits(onehot, x), x[perm])
    # small integers are exact in bf16 and fp64: compare with Python integers
    Wi = rng.integers(-8, 9, size=(E, H))
    xi = rng.integers(-50, 51, size=H)
    Wb = np.vectorize(bf16)(Wi.astype(float)).astype(np.uint16)
    want = [sum(int(Wi[e, j]) * int(xi[j]) for j in range(H)) for e in range(E)]
    assert list(om.router_logits(Wb, xi.astype(float))) == [float(v) for v in want]
    # T tokens at once equal T single calls; the shared gate is sigma of a one-row projection
    X = rng.standard_normal((3, H))
    Wr = synth.router_matrix(synth.TINY)[:E, :H].numpy().view(np.uint16)
    # (equal up to fp64 summation order: one matrix product against T matrix-vector products)
    assert np.allclose(om.router_logits(Wr, X), np.stack([om.router_logits(Wr, X[t]) for t in range(3)]),
                       rtol=1e-13, atol=1e-15)
    assert abs(om.shared_gate(Wr[0], X[0]) - float(om.sigmoid(om.router_logits(Wr[:1], X[0])[0]))) < 1e-15


def pin_dense_records():
    rng = np.random.default_rng(21)
    for bits, N, H in ((4, 5, 128), (2, 3, 192)):
        codes = rng.integers(0, 1 << bits, size=(N, H))
        scales = rng.choice([0.25, 0.5, 1.0, 2.0, 0.125], size=(N, H // 64))
        biases = rng.choice([-1.0, -0.5, 0.0, 0.25, 3.0], size=(N, H // 64))
        q = pack(codes, bits)
        sbw = np.array([[bf16(s) | (bf16(b) << 16) for s, b in zip(rs, rb)] for rs, rb in zip(scales, biases)],
                       dtype=np.uint32)
        rec = _up((q.shape[1] + sbw.shape[1]) * 4, 16) // 4
        words = np.zeros((N, rec), dtype=np.uint32)
        words[:, :q.shape[1]] = q
        words[:, q.shape[1]:q.shape[1] + sbw.shape[1]] = sbw
        W = om.dense_weights(words.reshape(-1), bits, N, H)
        want = codes * np.repeat(scales, 64, axis=1) + np.repeat(biases, 64, axis=1)
        assert np.array_equal(W, want)
        # integer inputs: every product and sum is exact in fp64
        x = rng.integers(-20, 21, size=H)
        res = rng.integers(-5, 6, size=N)
        exact = [sum(Fraction(float(want[r, c])) * int(x[c]) for c in range(H)) + int(res[r]) for r in range(N)]
        assert list(om.dense_matvec(W, x.astype(float), res.astype(float))) == [float(v) for v in exact]


def pin_rms_weight():
    rng = np.random.default_rng(22)
    h = rng.standard_normal(64)
    w = rng.standard_normal(64)
    assert np.array_equal(om.rms_norm(h, 1e-6, np.ones(64)), om.rms_norm(h, 1e-6))
    assert np.array_equal(om.rms_norm(h, 1e-6, 2 * w), 2 * om.rms_norm(h, 1e-6, w))
    # constant input c: every element is sign(c) / sqrt(1 + eps / c^2), times its weight
    c, eps = -0.75, 1e-6
    want = -1.0 / math.sqrt(1.0 + eps / (c * c)) * w
    assert np.allclose(om.rms_norm(np.full(64, c), eps, w), want, rtol=1e-14)


PINS = [pin_unpack_golden, pin_dequant_golden, pin_two_groups, pin_fma_identity,
        pin_group_decomposition, pin_random_blob_fields, pin_constant_rows, pin_route_bruteforce,
        pin_route_weights, pin_special_values, pin_zero_weight, pin_page_sizes,
        pin_layout_matches_generator, pin_block_closed_form, pin_stack_closed_form, pin_router_logits,
        pin_dense_records, pin_rms_weight]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ---------------------------------------------------------------------------
def _unpack_msb_first(words, bits):
    c = _ORIG["unpack_codes"](words, bits)
    per = 32 // bits
    return c.reshape(c.shape[:-1] + (-1, per))[..., ::-1].reshape(c.shape)


def _dequant_swapped(q_words, sb_words, bits):
    sbw = np.asarray(sb_words, dtype=np.uint32)
    return _ORIG["dequantize"](q_words, (sbw >> 16) | ((sbw & 0xFFFF) << 16), bits)


def _dequant_mod_group(q_words, sb_words, bits):
    q = om.unpack_codes(q_words, bits).astype(np.float64)
    sbw = np.asarray(sb_words, dtype=np.uint32)
    s, b = om.bf16_to_f64(sbw & 0xFFFF), om.bf16_to_f64(sbw >> 16)
    g = np.arange(q.shape[-1]) % sbw.shape[-1]
    return q * s[..., g] + b[..., g]


def _dequant_no_bias(q_words, sb_words, bits):
    sbw = np.asarray(sb_words, dtype=np.uint32)
    return _ORIG["dequantize"](q_words, sbw & 0xFFFF, bits)


def _ffn_swapped_swiglu(weights, x):
    wg, wu, wd = weights
    return wd @ (om.silu(wu @ x) * (wg @ x))


def _ffn_no_up(weights, x):
    wg, _, wd = weights
    return wd @ om.silu(wg @ x)


def _ffn_down_transposed(weights, x):
    wg, wu, wd = weights
    h = om.silu(wg @ x) * (wu @ x)
    return wd.T @ h if wd.shape[0] == wd.shape[1] else (wd.T @ h[: wd.shape[0]])


def _layout_gate_up_swapped(bits, hidden, inter):
    planes, nbytes = _ORIG["layout"](bits, hidden, inter)
    planes = dict(planes)
    planes["gate_q"], planes["up_q"] = planes["up_q"], planes["gate_q"]
    planes["gate_sb"], planes["up_sb"] = planes["up_sb"], planes["gate_sb"]
    return planes, nbytes


def _layout_down_parts_swapped(bits, hidden, inter):
    planes, nbytes = _ORIG["layout"](bits, hidden, inter)
    planes = dict(planes)
    (qo, qs, qr, qw), (so, ss, sr, sw) = planes["down_q"], planes["down_sb"]
    planes["down_q"], planes["down_sb"] = (so, qs, qr, qw), (qo, ss, sr, sw)
    return planes, nbytes


def _layout_up_rows_shifted(bits, hidden, inter):
    planes, nbytes = _ORIG["layout"](bits, hidden, inter)
    planes = dict(planes)
    off, stride, rows, wpr = planes["up_q"]
    planes["up_q"] = (off + stride, stride, rows, wpr) if rows > 1 else (off, stride, rows, wpr)
    return planes, nbytes


def _weights_down_row_major(blob, bits, hidden, inter):
    wg, wu, _ = _ORIG["expert_weights"](blob, bits, hidden, inter)
    q = om.unpack_codes(om.part_rows(blob, bits, hidden, inter, "down_q"), bits)   # [I][H], not transposed
    sbw = om.part_rows(blob, bits, hidden, inter, "down_sb").T
    return wg, wu, om.dequantize_codes(q.reshape(hidden, inter), sbw)


def _route_full_softmax(logits, k):
    l = np.asarray(logits, dtype=np.float64)
    ids = np.argsort(-l, kind="stable")[:k]
    e = np.exp(l - l.max())
    return ids, (e / e.sum())[ids]


def _route_ties_high(logits, k):
    l = np.asarray(logits, dtype=np.float64)
    ids = (len(l) - 1 - np.argsort(-l[::-1], kind="stable"))[:k]
    e = np.exp(l[ids] - l[ids].max())
    return ids, e / e.sum()


def _route_ascending(logits, k):
    ids, w = _ORIG["route"](logits, k)
    return ids[::-1], w[::-1]


def _gate_sign(wsg, x):
    return float(om.sigmoid(-(om.bf16_to_f64(wsg) @ np.asarray(x, dtype=np.float64))))


def _router_low_half(w, x):
    w = (np.asarray(w, dtype=np.uint32) & 0xFFFF).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64) @ w.T


def _router_rows_shifted(w, x):
    return np.roll(_ORIG["router_logits"](w, x), 1, axis=-1)


def _router_transposed(w, x):
    return np.asarray(x, dtype=np.float64) @ om.bf16_to_f64(w)


def _dense_scales_first(words, bits, n_rows, hidden):
    qw, sw, rw = om.dense_record_words(bits, hidden)
    rec = np.asarray(words, dtype=np.uint32).reshape(n_rows, rw)
    return om.dequantize(rec[:, sw:sw + qw], rec[:, :sw], bits)


def _dense_no_padding(words, bits, n_rows, hidden):
    qw, sw, _ = om.dense_record_words(bits, hidden)
    rec = np.asarray(words, dtype=np.uint32)[:n_rows * (qw + sw)].reshape(n_rows, qw + sw)
    return om.dequantize(rec[:, :qw], rec[:, qw:], bits)


def _rms_weight_ignored(h, eps, weight=None):
    return _ORIG["rms_norm"](h, eps)


def _combine_no_residual(residual, routed_y, weights, shared_y=None, g=None):
    return _ORIG["combine"](np.zeros_like(np.asarray(residual, dtype=np.float64)),
                            routed_y, weights, shared_y, g)


def _combine_unweighted_shared(residual, routed_y, weights, shared_y=None, g=None):
    return _ORIG["combine"](residual, routed_y, weights, shared_y, None if g is None else 1.0)


def _rms_eps_outside(h, eps, weight=None):
    h = np.asarray(h, dtype=np.float64)
    x = h / (np.sqrt(np.mean(h * h)) + eps)
    return x if weight is None else x * weight


def _rms_sum(h, eps, weight=None):
    h = np.asarray(h, dtype=np.float64)
    x = h / np.sqrt(np.sum(h * h) + eps)
    return x if weight is None else x * weight


_ORIG = {n: getattr(om, n) for n in ("unpack_codes", "dequantize", "route", "combine", "layout",
                                      "expert_weights", "router_logits", "rms_norm")}

MUTANTS = [
    ("unpack_codes", _unpack_msb_first),
    ("dequantize", _dequant_swapped),
    ("dequantize", _dequant_mod_group),
    ("dequantize", _dequant_no_bias),
    ("expert_ffn", _ffn_swapped_swiglu),
    ("expert_ffn", _ffn_no_up),
    ("expert_ffn", _ffn_down_transposed),
    ("layout", _layout_gate_up_swapped),
    ("layout", _layout_down_parts_swapped),
    ("layout", _layout_up_rows_shifted),
    ("expert_weights", _weights_down_row_major),
    ("route", _route_full_softmax),
    ("route", _route_ties_high),
    ("route", _route_ascending),
    ("shared_gate", _gate_sign),
    ("router_logits", _router_low_half),
    ("router_logits", _router_rows_shifted),
    ("router_logits", _router_transposed),
    ("dense_weights", _dense_scales_first),
    ("dense_weights", _dense_no_padding),
    ("rms_norm", _rms_weight_ignored),
    ("combine", _combine_no_residual),
    ("combine", _combine_unweighted_shared),
    ("rms_norm", _rms_eps_outside),
    ("rms_norm", _rms_sum),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=lambda v: getattr(v, "__name__", v))
def test_planted_mistakes(monkeypatch, name, mutant):
    monkeypatch.setattr(om, name, mutant)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {mutant.__name__}"
