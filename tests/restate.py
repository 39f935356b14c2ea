"""Independent restatements of the q6_K element map, used to pin the oracle.

The pages describe the same element -> byte map three ways. The oracle
implements the per-element form ("r38 -- q6_K BT-style raw-byte mma kernel",
Sec. 3.2). This module restates the other two, in numpy, so that the oracle's
decode is checked against descriptions it does not share:

* ``decode_pairs``: the load-time expander of "r53 -- q6_K bundle: W_exp
  pre-expansion plane" Sec. 3.2: one (ql byte, qh byte) pair yields the two
  elements r and r+64 of a 128-element half, from the low and the high nibble
  of the ql byte and two 2-bit fields of the qh byte four bits apart.
* ``decode_groups``: the 16-element group closed form of "r41 -- q6_K B-expand
  widened to uint4 group loads" Sec. 3.2: for an even 32-chunk base ``cbase``
  and group ``gg`` (0..3) of a 64-element window, a 16-byte ql run, a 16-byte
  qh run, one nibble shift and one 2-bit field shift serve all 16 elements.

``encode`` is the inverse of ``decode_pairs`` (codes -> ql/qh bytes) so tests
can build blocks with chosen codes.
"""
from __future__ import annotations

import numpy as np

QK = 256
BLOCK_BYTES = 210


def decode_pairs(blk: np.ndarray) -> np.ndarray:
    """Codes 0..63 of one 210-byte block, by (ql, qh) byte pairs."""
    blk = np.asarray(blk, dtype=np.uint8)
    codes = np.empty(QK, dtype=np.int32)
    for half in range(2):
        r = np.arange(64)
        ql = blk[64 * half + r].astype(np.int32)
        qh = blk[128 + 32 * half + (r % 32)].astype(np.int32)
        first = 2 * (r // 32)               # field of element r; r+64 uses first+4
        codes[128 * half + r] = (ql & 0xF) | (((qh >> first) & 3) << 4)
        codes[128 * half + r + 64] = (ql >> 4) | (((qh >> (first + 4)) & 3) << 4)
    return codes


def decode_groups(blk: np.ndarray) -> np.ndarray:
    """Codes 0..63 of one block, by 16-element groups of a 64-element window."""
    blk = np.asarray(blk, dtype=np.uint8)
    codes = np.empty(QK, dtype=np.int32)
    for cbase in (0, 2, 4, 6):              # window = chunks cbase, cbase+1
        it0 = (cbase >> 2) & 1
        nib = ((cbase >> 1) & 1) * 4
        for gg in range(4):
            qlrun = blk[it0 * 64 + gg * 16: it0 * 64 + gg * 16 + 16].astype(np.int32)
            qhrun = blk[128 + it0 * 32 + (gg & 1) * 16:
                        128 + it0 * 32 + (gg & 1) * 16 + 16].astype(np.int32)
            fld = nib + ((gg >> 1) & 1) * 2
            e0 = cbase * 32 + gg * 16
            codes[e0:e0 + 16] = ((qlrun >> nib) & 0xF) | (((qhrun >> fld) & 3) << 4)
    return codes


def encode(codes: np.ndarray) -> np.ndarray:
    """ql[128] + qh[64] bytes (192 bytes) holding the 256 given 6-bit codes."""
    codes = np.asarray(codes, dtype=np.int32)
    assert codes.shape == (QK,) and codes.min() >= 0 and codes.max() < 64
    out = np.zeros(192, dtype=np.uint8)
    for half in range(2):
        c = codes[128 * half: 128 * half + 128]
        out[64 * half: 64 * half + 64] = (c[0:64] & 0xF) | ((c[64:128] & 0xF) << 4)
        qh = np.zeros(32, dtype=np.int32)
        for f in range(4):
            qh |= ((c[32 * f: 32 * f + 32] >> 4) & 3) << (2 * f)
        out[128 + 32 * half: 128 + 32 * half + 32] = qh
    return out


def make_block(codes, sc, d_f16_bits: int) -> np.ndarray:
    """A full 210-byte block from codes[256], sc[16] (int) and f16 bits of d."""
    blk = np.zeros(BLOCK_BYTES, dtype=np.uint8)
    blk[0:192] = encode(np.asarray(codes))
    blk[192:208] = np.asarray(sc, dtype=np.int64).astype(np.int8).view(np.uint8)
    blk[208] = d_f16_bits & 0xFF
    blk[209] = (d_f16_bits >> 8) & 0xFF
    return blk


def dequantize(raw: np.ndarray, M: int, K: int) -> np.ndarray:
    """f64 W[M, K] = d * sc[sub] * (code - 32), from decode_pairs and numpy's f16."""
    nsb = K // QK
    blocks = np.asarray(raw, dtype=np.uint8).reshape(M * nsb, BLOCK_BYTES)
    W = np.empty((M * nsb, QK), dtype=np.float64)
    for i, blk in enumerate(blocks):
        v = decode_pairs(blk) - 32
        d = float(blk[208:210].view(np.float16)[0])
        sc = blk[192:208].view(np.int8).astype(np.float64)
        W[i] = d * np.repeat(sc, 16) * v
    return W.reshape(M, K)


def int_values(raw: np.ndarray, M: int, K: int) -> np.ndarray:
    """Centered int64 values [M, K] from decode_pairs."""
    nsb = K // QK
    blocks = np.asarray(raw, dtype=np.uint8).reshape(M * nsb, BLOCK_BYTES)
    return np.stack([decode_pairs(b) - 32 for b in blocks]).astype(np.int64).reshape(M, K)
