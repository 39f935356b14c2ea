"""Pins of the CPU oracle: checks against what the pages and mathematics fix.

Every pin is a function ``pin_x(orc)`` that raises ``AssertionError`` when the
oracle build ``orc`` disagrees with something other than itself: a value the
pages print (fixtures under ``tests/golden/``), an independent restatement of
the element map from another page (``restate.py``), a library routine
(numpy's binary16 decode, integer matmul), exact rational arithmetic, or an
invariant of the method. ``test_oracle_pins.py`` runs each pin on the real
oracle and runs the whole list on builds with one planted mistake each, to
show that every such mistake fails at least one pin.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import restate
from q6_int8_mmq_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F16_ONE = 0x3C00


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out[k] = [int(x) for x in v] if len(v) > 1 else int(v[0])
    return out


def _all32_block(d_bits=F16_ONE, sc=None):
    return restate.make_block(np.full(256, 32), np.zeros(16) if sc is None else sc, d_bits)


def _rand_raw(seed, M, K):
    return synth.q6k_raw_weights(seed, M, K)


# ------------------------------------------------------------------ decode --

def pin_block_layout(orc):
    """Offsets from the page's table: decode reads only ql and qh (bytes 0..191);
    sc byte s feeds dsc of sub-block s alone; the d bytes feed all sixteen."""
    g = _golden("q6k_block_layout.txt")
    assert g["total"] == 210 and g["d"][0] + g["d"][1] == 210
    blk = _rand_raw(11, 1, 256)[0].copy()
    blk[208:210] = np.array([0x00, 0x3C], np.uint8)          # d = 1.0
    sc = blk[192:208].view(np.int8)
    base = orc.decode_block(blk)
    dsc0 = orc.dsc(blk, 1, 256)[0]
    q_end = g["qh"][0] + g["qh"][1]
    for byte in range(210):
        b2 = blk.copy()
        b2[byte] ^= 0x01
        dec_changed = not np.array_equal(orc.decode_block(b2), base)
        assert dec_changed == (byte < q_end), f"decode vs byte {byte}"
        changed = list(np.nonzero(orc.dsc(b2, 1, 256)[0] != dsc0)[0])
        if g["sc"][0] <= byte < g["sc"][0] + g["sc"][1]:
            assert changed == [byte - g["sc"][0]], f"sc byte {byte}"
        elif byte >= g["d"][0]:
            assert changed == list(np.nonzero(sc != 0)[0]), f"d byte {byte}"
        else:
            assert changed == [], f"dsc vs byte {byte}"


def pin_elem70(orc):
    """The page's worked element: ql/qh bytes, sub-block and chunk of element 70."""
    g = _golden("q6k_elem70.txt")
    e = g["element"]
    blk = _all32_block()
    # high nibble of ql[6] := 5, field at qh[6] bits 4..5 := 1  ->  code 5 | 1<<4
    qlb, qh = g["ql_byte"], 128 + g["qh_byte"]
    blk[qlb] = (int(blk[qlb]) & (0xFF ^ (0xF << g["ql_shift"]))) | (5 << g["ql_shift"])
    blk[qh] = (int(blk[qh]) & (0xFF ^ (3 << g["qh_shift"]))) | (1 << g["qh_shift"])
    dec = orc.decode_block(blk).astype(np.int64)
    want = np.zeros(256, dtype=np.int64)
    want[e] = (5 | (1 << 4)) - 32
    assert np.array_equal(dec, want), "element 70 byte positions"
    # sub-block and chunk: only sc[subblock] and da[chunk] may scale element 70
    sc = np.arange(16) + 10
    blk[192:208] = sc.astype(np.int8).view(np.uint8)
    xq = np.zeros((1, 256), dtype=np.int8)
    xq[0, e] = 7
    assert e // 32 == g["chunk"] and e % 32 == g["chunk_offset"] and e // 16 == g["subblock"]
    da = (2.0 ** -np.arange(8)).astype(np.float32)[None, :]
    Y = orc.mmq(blk, 1, 256, xq, da)
    want_y = 1.0 * sc[g["subblock"]] * float(da[0, g["chunk"]]) * (-11) * 7
    assert Y[0, 0] == want_y, (Y[0, 0], want_y)


def pin_restatements(orc):
    """Per-element form (oracle) == pair form (r53) == group form (r41), all 256 positions."""
    raw = _rand_raw(12, 64, 256)
    for blk in raw:
        dec = orc.decode_block(blk).astype(np.int64) + 32
        assert np.array_equal(dec, restate.decode_pairs(blk)), "pair form"
        assert np.array_equal(dec, restate.decode_groups(blk)), "group form"


def pin_bijection(orc):
    """Every ql/qh bit feeds exactly one element; every element has 4+2 bits."""
    blk = _rand_raw(13, 1, 256)[0].copy()
    base = orc.decode_block(blk)
    hits = np.zeros(256, dtype=np.int64)
    for byte in range(192):
        for bit in range(8):
            b2 = blk.copy()
            b2[byte] ^= (1 << bit)
            diff = np.nonzero(orc.decode_block(b2) != base)[0]
            assert diff.size == 1, f"bit {byte}.{bit} feeds {diff.size} elements"
            hits[diff[0]] += 1
    assert np.all(hits == 6)


def pin_all32(orc):
    """ql 0x00 / qh 0xAA encodes code 32 everywhere: every value and Y are zero."""
    blk = np.zeros(210, dtype=np.uint8)
    blk[128:192] = 0xAA
    blk[192:208] = np.arange(16, dtype=np.int8).view(np.uint8) + 1
    blk[208:210] = np.array([0x00, 0x3C], dtype=np.uint8)
    assert np.all(orc.decode_block(blk) == 0)
    raw = np.tile(blk, (4, 2))                    # M=4, K=512
    X = synth.activations(14, 3, 512)
    xq, da = orc.quantize(X)
    assert np.all(orc.mmq(raw, 4, 512, xq, da) == 0.0)


def pin_d_zero(orc):
    raw = _rand_raw(15, 4, 512).copy().reshape(-1, 210)
    raw[:, 208:210] = 0
    X = synth.activations(15, 3, 512)
    xq, da = orc.quantize(X)
    assert np.all(orc.mmq(raw.reshape(4, -1), 4, 512, xq, da) == 0.0)


# ---------------------------------------------------------------- f16, dsc --

def pin_f16(orc):
    """Exact binary16 decode (subnormals included) == numpy's float16 -> float64."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(x)) for x in h])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def pin_dsc(orc):
    """dsc = f32(d) * sc exactly; hand values at the ends of both ranges."""
    cases = [(0x0001, -128, -(2.0 ** -17)), (0x3C00, 127, 127.0),
             (0x7BFF, -128, -65504.0 * 128), (0x03FF, 3, 3 * 1023 * 2.0 ** -24),
             (0x8400, 5, -5 * 2.0 ** -14)]
    for bits, sc, want in cases:
        s = np.zeros(16)
        s[7] = sc
        blk = _all32_block(bits, s)
        assert orc.dsc(blk, 1, 256)[0, 7] == np.float32(want), (bits, sc)
    raw = _rand_raw(16, 8, 512)
    got = orc.dsc(raw, 8, 512)
    blocks = raw.reshape(-1, 210)
    d = blocks[:, 208:210].copy().view(np.float16).astype(np.float32)
    sc = blocks[:, 192:208].view(np.int8).astype(np.float32)
    assert np.array_equal(got.reshape(-1, 16), d * sc)


def pin_wexp(orc):
    raw = _rand_raw(17, 6, 768)
    w = orc.wexp(raw, 6, 768)
    assert np.array_equal(w.astype(np.int64), restate.int_values(raw, 6, 768))
    assert w.min() >= -32 and w.max() <= 31


# -------------------------------------------------------------------- GEMM --

def pin_bruteforce(orc):
    """Dequantise both sides to f64 (restated decode, numpy f16) and matmul."""
    M, K, N = 8, 512, 5
    raw = _rand_raw(18, M, K).copy().reshape(-1, 210)
    raw[0, 192] = 0x80                                    # sc = -128
    raw[1, 208:210] = np.array([0x07, 0x00], np.uint8)    # subnormal d
    raw = raw.reshape(M, -1)
    X = synth.activations(18, N, K)
    xq, da = orc.quantize(X)
    W = restate.dequantize(raw, M, K)
    Xd = xq.astype(np.float64) * np.repeat(da.astype(np.float64), 32, axis=1)
    ref = Xd @ W.T
    Y = orc.mmq(raw, M, K, xq, da)
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def pin_integer_case(orc):
    """d = 1, sc = 1, da = 1: Y is the integer GEMM of (q - 32) and xq."""
    M, K, N = 6, 512, 4
    raw = _rand_raw(19, M, K).copy().reshape(-1, 210)
    raw[:, 192:208] = 1
    raw[:, 208:210] = np.array([0x00, 0x3C], np.uint8)
    raw = raw.reshape(M, -1)
    xq = synth.uniform_bytes(19, N * K).view(np.int8).reshape(N, K).copy()
    xq[xq == -128] = -127
    da = np.ones((N, K // 32), dtype=np.float32)
    ref = xq.astype(np.int64) @ restate.int_values(raw, M, K).T
    Y = orc.mmq(raw, M, K, xq, da)
    assert np.array_equal(Y, ref.astype(np.float64))


def pin_partials(orc):
    M, K, N = 5, 512, 3
    raw = _rand_raw(20, M, K)
    xq = synth.uniform_bytes(20, N * K).view(np.int8).reshape(N, K).copy()
    xq[xq == -128] = 127
    da = np.ones((N, K // 32), dtype=np.float32)
    _, P = orc.mmq(raw, M, K, xq, da, partials=True)
    V = restate.int_values(raw, M, K)
    ref = np.einsum("nsk,msk->nms", xq.astype(np.int64).reshape(N, K // 16, 16),
                    V.reshape(M, K // 16, 16))
    assert np.array_equal(P.astype(np.int64), ref)


def pin_subblock_removal(orc):
    """sc = 0 in one sub-block removes exactly that sub-block's contribution."""
    K, N = 512, 3
    raw = _rand_raw(21, 1, K).copy().reshape(-1, 210)
    X = synth.activations(21, N, K)
    xq, da = orc.quantize(X)
    b, s = 1, 9
    raw0 = raw.copy()
    raw0[b, 192 + s] = 0
    y_sc0 = orc.mmq(raw0.reshape(1, -1), 1, K, xq, da)
    xq0 = xq.copy()
    xq0[:, 256 * b + 16 * s: 256 * b + 16 * s + 16] = 0
    y_x0 = orc.mmq(raw.reshape(1, -1), 1, K, xq0, da)
    assert np.array_equal(y_sc0, y_x0)
    assert not np.array_equal(y_sc0, orc.mmq(raw.reshape(1, -1), 1, K, xq, da))


def pin_linearity(orc):
    """Integer partials are additive in xq (exact)."""
    M, K, N = 4, 512, 3
    raw = _rand_raw(22, M, K)
    a = (synth.uniform_bytes(22, N * K).view(np.int8) // 2).reshape(N, K)
    b = (synth.uniform_bytes(23, N * K).view(np.int8) // 2).reshape(N, K)
    da = np.ones((N, K // 32), dtype=np.float32)
    _, Pa = orc.mmq(raw, M, K, a, da, partials=True)
    _, Pb = orc.mmq(raw, M, K, b, da, partials=True)
    _, Pab = orc.mmq(raw, M, K, (a + b).astype(np.int8), da, partials=True)
    assert np.array_equal(Pab.astype(np.int64), Pa.astype(np.int64) + Pb)


def pin_pow2_scaling(orc):
    """X -> 2^k X: xq unchanged, da doubled k times exactly, Y scaled by 2^k exactly."""
    M, K, N = 4, 512, 3
    raw = _rand_raw(24, M, K)
    X = synth.activations(24, N, K)
    xq, da = orc.quantize(X)
    Y = orc.mmq(raw, M, K, xq, da)
    for k in (3, -5):
        xq2, da2 = orc.quantize((X * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(xq2, xq)
        assert np.array_equal(da2, (da * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(orc.mmq(raw, M, K, xq2, da2), Y * 2.0 ** k)


def pin_single_block_closed_form(orc):
    """One super-block with one non-32 code per sub-block, summed exactly."""
    rng_codes = synth.uniform_bytes(25, 64)
    pos = [16 * s + int(rng_codes[s]) % 16 for s in range(16)]
    amp = [int(rng_codes[16 + s]) % 31 + 1 for s in range(16)]       # code 32 + amp
    amp = [a if s % 3 else -a for s, a in enumerate(amp)]
    codes = np.full(256, 32)
    for s in range(16):
        codes[pos[s]] = 32 + amp[s]
    sc = [int(v) for v in synth.uniform_bytes(26, 16).view(np.int8)]
    d_bits = 0x1A3D                                                    # 0.0031...
    blk = restate.make_block(codes, sc, d_bits)
    N = 2
    xq = synth.uniform_bytes(27, N * 256).view(np.int8).reshape(N, 256).copy()
    xq[xq == -128] = -1
    da = np.array([[2.0 ** -(c + 1) * (1 + n) for c in range(8)] for n in range(N)],
                  dtype=np.float32)
    d = Fraction(float(np.array([d_bits], np.uint16).view(np.float16)[0]))
    Y = orc.mmq(blk, 1, 256, xq, da)
    for n in range(N):
        want = sum(d * sc[s] * Fraction(float(da[n, pos[s] // 32])) * amp[s] * int(xq[n, pos[s]])
                   for s in range(16))
        assert abs(Y[n, 0] - float(want)) <= 1e-15 * abs(float(want)) + 1e-300, (n, Y[n, 0], float(want))


# -------------------------------------------------------------- quantizer --

def pin_quantizer_properties(orc):
    N, K = 16, 1024
    X = synth.activations(28, N, K, outlier_frac=0.05)
    X[3, 64:96] = 0.0                             # an all-zero block
    X[4, 0:32] = np.float32(1e-30)                # tiny but nonzero
    xq, da = orc.quantize(X)
    assert xq.min() >= -127 and xq.max() <= 127
    xb = X.reshape(N, K // 32, 32).astype(np.float64)
    qb = xq.reshape(N, K // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    assert np.all(da[amax == 0] == 0) and np.all(qb[amax == 0] == 0)
    nz = amax > 0
    # da = amax/127 up to one f32 rounding
    assert np.all(np.abs(da[nz].astype(np.float64) * 127 - amax[nz]) <= amax[nz] * 2.0 ** -23)
    # the largest-magnitude element of every block maps to +-127
    arg = np.abs(xb).argmax(axis=2)
    top = np.take_along_axis(qb, arg[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top[nz]) == 127)
    # every code is a nearest integer of x/da (to within the f32 quotient's rounding)
    err = np.abs(xb - da[..., None].astype(np.float64) * qb)
    assert np.all(err[nz] <= da[nz][:, None] * (0.5 + 2.0 ** -20))


def pin_quantizer_rounding(orc):
    """Halfway quotients round away from zero: amax = 127 makes da = 1 exactly."""
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 127.0
    x[0, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, 3.49, -3.51, 126.5]
    xq, da = orc.quantize(x)
    assert da[0, 0] == 1.0
    assert list(xq[0, :9]) == [127, 3, -3, 1, -1, 2, 3, -4, 127]


# -------------------------------------------------------------------- q4_K --
# The q4_K line ("r18: Load-time B pre-expansion", Sec. 1 and 3.2; the
# two-term rescale of "r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2).

def _q4k_raw(seed, M, K):
    return synth.q4k_raw_weights(seed, M, K)


def _q4k_values(orc, s12):
    return [orc.q4k_scale_min(s12, j) for j in range(8)]


def pin_q4k_scale_example(orc):
    """The hand-worked example of the scale/min packing reading (golden)."""
    g = _golden("q4k_scale_min.txt")
    vals = _q4k_values(orc, np.array(g["bytes"], np.uint8))
    assert [v[0] for v in vals] == g["scales"]
    assert [v[1] for v in vals] == g["mins"]


def pin_q4k_scale_bijection(orc):
    """Every one of the 96 bits of the 12 packed bytes moves exactly one of
    the sixteen 6-bit values by exactly one power of two, and each (value,
    bit) pair is reached by exactly one byte bit."""
    rng = np.random.default_rng(41)
    for _ in range(4):
        s12 = rng.integers(0, 256, 12).astype(np.uint8)
        base = np.array(_q4k_values(orc, s12)).T.reshape(16)    # 8 scales, then 8 mins
        assert np.all((base >= 0) & (base < 64))
        hit = set()
        for byte in range(12):
            for bit in range(8):
                s2 = s12.copy()
                s2[byte] ^= np.uint8(1 << bit)
                diff = np.array(_q4k_values(orc, s2)).T.reshape(16) - base
                nz = np.nonzero(diff)[0]
                assert len(nz) == 1, (byte, bit)
                step = abs(int(diff[nz[0]]))
                assert step & (step - 1) == 0 and step < 64
                hit.add((int(nz[0]), step.bit_length() - 1))
        assert len(hit) == 96


def pin_q4k_nibble_map(orc):
    """The element map of the page's in-loop B expansion, restated: for
    nibble pair p the 32 bytes at 16 + 32 p give sub-block 2 p (low nibbles)
    and 2 p + 1 (high nibbles), element-ordered, raw values 0..15."""
    for blk in _q4k_raw(42, 3, 256):
        codes = orc.q4k_decode_block(blk)[0]
        want = []
        for p in range(4):
            run = blk[16 + 32 * p: 16 + 32 * p + 32]
            want += list(run & 0x0F) + list(run >> 4)
        assert np.array_equal(codes, np.array(want, np.uint8))


def pin_q4k_block_layout(orc):
    """d at bytes 0-1, dmin at 2-3, the packed scales at 4-15 and the nibbles
    at 16-143: flipping a byte changes only what lives there."""
    blk = _q4k_raw(43, 1, 256)[0].copy()
    c0, s0, m0, d0, n0 = orc.q4k_decode_block(blk)
    for byte in range(144):
        b2 = blk.copy()
        b2[byte] ^= 0x01
        c, s, m, d, n = orc.q4k_decode_block(b2)
        changed = (not np.array_equal(c, c0), not (np.array_equal(s, s0) and np.array_equal(m, m0)),
                   d != d0, n != n0)
        want = (byte >= 16, 4 <= byte < 16, byte < 2, 2 <= byte < 4)
        assert changed == want, byte


def _q4k_dequant(orc, raw, M, K):
    """Dequantised weights d*sc*q - dmin*m in f64 from the oracle's block decode."""
    W = np.empty((M, K))
    for m in range(M):
        for b in range(K // 256):
            codes, sc, mn, d, dmin = orc.q4k_decode_block(raw[m, 144 * b: 144 * (b + 1)])
            c = np.arange(256) // 32
            W[m, 256 * b: 256 * (b + 1)] = d * sc[c] * codes - dmin * mn[c]
    return W


def pin_q4k_bruteforce(orc):
    """Dequantise both sides to f64 and multiply (numpy): the GEMM agrees."""
    M, K, N = 7, 512, 5
    raw = _q4k_raw(44, M, K)
    xq, da = orc.quantize(synth.activations(45, N, K, outlier_frac=0.05))
    X = xq.astype(np.float64) * np.repeat(da.astype(np.float64), 32, axis=1)
    Yb = X @ _q4k_dequant(orc, raw, M, K).T
    Y = orc.q4k_mmq(raw, M, K, xq, da)
    assert np.max(np.abs(Y - Yb)) <= 1e-12 * np.max(np.abs(Yb))


def pin_q4k_integer_case(orc):
    """d = 1, dmin = 0, every scale 1 and integer activations with da = 1
    reduce the GEMM to the int64 matmul of the nibbles and xq; the debug
    partials are the per-32 sums of that product."""
    M, K, N = 6, 512, 4
    raw = _q4k_raw(46, M, K).reshape(-1, 144).copy()
    raw[:, 0:2] = [0x00, 0x3C]                     # d = 1.0
    raw[:, 2:4] = 0                                # dmin = 0
    raw[:, 4:8] = 1                                # scales 0..3 = 1, top bits 0
    raw[:, 8:12] = 0                               # mins 0..3 = 0, top bits 0
    raw[:, 12:16] = 0x01                           # scales 4..7 = 1, mins 4..7 = 0
    raw = raw.reshape(M, -1)
    rng = np.random.default_rng(47)
    X = rng.integers(-127, 128, size=(N, K)).astype(np.float32)
    X[:, ::32] = 127.0                             # amax 127 in every block: da = 1
    xq, da = orc.quantize(X)
    assert np.all(da == 1.0) and np.array_equal(xq, X.astype(np.int8))
    Q = np.stack([np.concatenate([orc.q4k_decode_block(raw[m, 144 * b: 144 * (b + 1)])[0]
                                  for b in range(K // 256)]) for m in range(M)]).astype(np.int64)
    Y, P = orc.q4k_mmq(raw, M, K, xq, da, partials=True)
    assert np.array_equal(Y, (xq.astype(np.int64) @ Q.T).astype(np.float64))
    Pw = (xq.astype(np.int64)[:, None, :] * Q[None]).reshape(N, M, K // 32, 32).sum(-1)
    assert np.array_equal(P, Pw)


def pin_q4k_min_term(orc):
    """All nibbles 0 leave only the min term: Y = -sum dmin*m*da*sum(xq) over
    the sub-blocks (closed form), and the partials are 0."""
    M, K, N = 3, 512, 4
    raw = _q4k_raw(48, M, K).reshape(-1, 144).copy()
    raw[:, 16:] = 0
    raw = raw.reshape(M, -1)
    xq, da = orc.quantize(synth.activations(49, N, K))
    S = xq.astype(np.int64).reshape(N, K // 32, 32).sum(-1)
    want = np.zeros((N, M))
    for m in range(M):
        for b in range(K // 256):
            _, _, mn, _, dmin = orc.q4k_decode_block(raw[m, 144 * b: 144 * (b + 1)])
            for j in range(8):
                c = 8 * b + j
                want[:, m] -= dmin * mn[j] * da[:, c].astype(np.float64) * S[:, c]
    Y, P = orc.q4k_mmq(raw, M, K, xq, da, partials=True)
    assert np.all(P == 0)
    assert np.max(np.abs(Y - want)) <= 1e-12 * np.max(np.abs(want))


PINS = [pin_block_layout, pin_elem70, pin_restatements, pin_bijection, pin_all32,
        pin_d_zero, pin_f16, pin_dsc, pin_wexp, pin_bruteforce, pin_integer_case,
        pin_partials, pin_subblock_removal, pin_linearity, pin_pow2_scaling,
        pin_single_block_closed_form, pin_quantizer_properties, pin_quantizer_rounding,
        pin_q4k_scale_example, pin_q4k_scale_bijection, pin_q4k_nibble_map,
        pin_q4k_block_layout, pin_q4k_bruteforce, pin_q4k_integer_case, pin_q4k_min_term]


def failing_pins(orc):
    """Names of the pins this oracle build fails."""
    bad = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception:           # any failure (assertion or crash) counts
            bad.append(pin.__name__)
    return bad
