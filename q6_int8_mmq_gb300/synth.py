"""Seeded synthetic inputs for the q6_K x int8 GEMM.

This module produces raw GGUF-layout q6_K weight bytes and f32 activation
matrices from a counter-based generator. It holds none of the method's own
arithmetic: no decode, no quantization, no scaling. The test-suite (which
feeds the CPU oracle) and the benchmark (which feeds the CUDA library) both
draw their inputs from here, so the two sides see identical bytes.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used in counter mode,
``x_i = mix64(seed + (i + 1) * 0x9E3779B97F4A7C15)``, with Box-Muller for
normal deviates.

Workload recipe (value distributions of the tiny q6_K x int8 GEMM case, reused
by every workload):
  * q6_K super-block of 210 bytes: ql[128] and qh[64] uniform random bytes
    (so every 6-bit code is uniform on 0..63 whatever the byte map), sc[16]
    uniform int8 on [-128, 127], d = float16(|N(0,1)| * 2e-3) at bytes
    208..209 (little endian).
  * activations: f32 ~ N(0,1); optionally a seeded set of outlier channels
    (columns of X) multiplied by 20.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK = 256          # elements per q6_K super-block
BLOCK_BYTES = 210  # bytes per raw q6_K super-block

# Base seeds per workload; layer l of the 32-layer sweep uses SWEEP_SEED + l.
WORKLOAD_SEED = {
    "tiny": 0x51360000,
    "attn_v": 0x51360001,
    "ffn_down": 0x51360002,
    "skinny": 0x51360003,
    "sweep": 0x51360004,
    "pages_ffn_down": 0x51360005,
    "pages_attn_v": 0x51360006,
    "pages_ffn_up": 0x51360007,
}
SWEEP_SEED = 0x51364000

# Workload shapes: (M weight rows, K, N tokens).
WORKLOADS = {
    "tiny": dict(M=256, K=512, N=8, outlier_frac=0.0),
    "attn_v": dict(M=4096, K=4096, N=512, outlier_frac=0.0),
    "ffn_down": dict(M=4096, K=11008, N=3314, outlier_frac=0.01),
    # the shapes the pages measure (a Qwen2-class 7B: hidden 3584, FFN 18944,
    # 512-wide grouped V projection) at their ~3325-token prefill
    "pages_ffn_down": dict(M=3584, K=18944, N=3325, outlier_frac=0.01),
    "pages_attn_v": dict(M=512, K=3584, N=3325, outlier_frac=0.0),
    # the pages' model is q4_k_m: its FFN gate/up projections (18944 x 3584)
    # are q4_K weights (q4k_workload)
    "pages_ffn_up": dict(M=18944, K=3584, N=3325, outlier_frac=0.01),
}
SKINNY_SHAPES = {"ffn_down": (4096, 11008), "attn_v": (4096, 4096)}
SKINNY_N = (1, 2, 4, 16)
SWEEP_LAYERS = 32
SWEEP_N = 3314


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of the SplitMix64 stream for ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GOLDEN
        return _mix(z)


def substream(seed: int, tag: int) -> int:
    """A derived seed for an independent stream (one draw of ``seed`` at ``tag``)."""
    return int(splitmix64(seed, 1, offset=tag)[0])


def uniform_bytes(seed: int, n: int) -> np.ndarray:
    words = splitmix64(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def uniform01(seed: int, n: int) -> np.ndarray:
    """Uniform doubles on the open interval (0, 1): 53 high bits, half-ulp offset."""
    z = splitmix64(seed, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def _uniform01_at(seed: int, n: int, offset: int) -> np.ndarray:
    z = splitmix64(seed, n, offset)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int, chunk: int = 1 << 18) -> np.ndarray:
    """Standard normal deviates by Box-Muller (cosine branch), float64.

    Deviate i uses draws 2i and 2i+1 of the stream; the work is done in
    cache-sized chunks, which changes nothing in the values.
    """
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        u = _uniform01_at(seed, 2 * m, 2 * s)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return out


# ---------------------------------------------------------------- weights ---

def q6k_raw_weights(seed: int, M: int, K: int) -> np.ndarray:
    """Raw q6_K weight matrix, GGUF byte layout: uint8 [M, (K/256)*210].

    Block byte map (per super-block): ql @0..127, qh @128..191,
    sc (int8) @192..207, d (f16, little endian) @208..209.
    """
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    nblk = M * (K // QK)
    blk = np.empty((nblk, BLOCK_BYTES), dtype=np.uint8)
    blk[:, 0:192] = uniform_bytes(substream(seed, 1), nblk * 192).reshape(nblk, 192)
    blk[:, 192:208] = uniform_bytes(substream(seed, 2), nblk * 16).reshape(nblk, 16)
    d = (np.abs(normal(substream(seed, 3), nblk)) * 2e-3).astype(np.float16)
    blk[:, 208:210] = d.view(np.uint8).reshape(nblk, 2)
    return blk.reshape(M, (K // QK) * BLOCK_BYTES)


Q4K_BLOCK_BYTES = 144


def q4k_raw_weights(seed: int, M: int, K: int) -> np.ndarray:
    """Raw q4_K weight matrix, GGUF byte layout: uint8 [M, (K/256)*144].

    Block byte map (per super-block): d (f16) @0..1, dmin (f16) @2..3, the 12
    bytes of packed 6-bit scales and mins @4..15, the 128 nibble bytes
    @16..143. Nibbles, scales and mins are uniform (uniform bytes give
    uniform 4-bit and 6-bit values under any bit packing), d and dmin are
    f16(|N(0,1)| * 2e-3) like the q6_K recipe's d.
    """
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    nblk = M * (K // QK)
    blk = np.empty((nblk, Q4K_BLOCK_BYTES), dtype=np.uint8)
    d = (np.abs(normal(substream(seed, 3), nblk)) * 2e-3).astype(np.float16)
    dmin = (np.abs(normal(substream(seed, 4), nblk)) * 2e-3).astype(np.float16)
    blk[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
    blk[:, 2:4] = dmin.view(np.uint8).reshape(nblk, 2)
    blk[:, 4:144] = uniform_bytes(substream(seed, 1), nblk * 140).reshape(nblk, 140)
    return blk.reshape(M, (K // QK) * Q4K_BLOCK_BYTES)


# ------------------------------------------------------------ activations ---

def outlier_channels(seed: int, K: int, frac: float) -> np.ndarray:
    """Indices of round(frac*K) seeded channels (a seeded permutation prefix)."""
    cnt = int(round(frac * K))
    if cnt == 0:
        return np.zeros(0, dtype=np.int64)
    keys = splitmix64(substream(seed, 5), K)
    return np.sort(np.argsort(keys, kind="stable")[:cnt])


def activations(seed: int, N: int, K: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    """f32 X[N, K] ~ N(0,1), with optional outlier channels scaled up."""
    x = normal(substream(seed, 4), N * K).astype(np.float32).reshape(N, K)
    ch = outlier_channels(seed, K, outlier_frac)
    if ch.size:
        x[:, ch] *= np.float32(outlier_scale)
    return x


# -------------------------------------------------------------- workloads ---

def workload(name: str):
    """(raw q6_K weights, f32 activations, shape dict) for a named workload."""
    cfg = WORKLOADS[name]
    seed = WORKLOAD_SEED[name]
    raw = q6k_raw_weights(seed, cfg["M"], cfg["K"])
    x = activations(seed, cfg["N"], cfg["K"], cfg["outlier_frac"])
    return raw, x, dict(cfg)


Q4K_SEED = 0x51361401


def q4k_workload(name: str = "ffn_down"):
    """(raw q4_K weights, f32 activations, shape dict): the named workload's
    shape and activation stream with q4_K weights in place of q6_K."""
    cfg = WORKLOADS[name]
    x = activations(WORKLOAD_SEED[name], cfg["N"], cfg["K"], cfg["outlier_frac"])
    seed = Q4K_SEED ^ (WORKLOAD_SEED[name] - WORKLOAD_SEED["ffn_down"])
    return q4k_raw_weights(seed, cfg["M"], cfg["K"]), x, dict(cfg)


def skinny_workload(weight: str, n: int):
    M, K = SKINNY_SHAPES[weight]
    seed = WORKLOAD_SEED["skinny"] + (0x100 if weight == "attn_v" else 0)
    raw = q6k_raw_weights(seed, M, K)
    x = activations(substream(seed, 0x40 + n), n, K)
    return raw, x, dict(M=M, K=K, N=n)


def sweep_layer(layer: int):
    """Layer ``layer`` of the 32-layer 7B-shape sweep: (raw_attn_v, raw_ffn_down)."""
    seed = SWEEP_SEED + layer
    return (q6k_raw_weights(substream(seed, 0x10), 4096, 4096),
            q6k_raw_weights(substream(seed, 0x11), 4096, 11008))


def sweep_activations():
    """The two f32 activation streams of the sweep: X_v [3314,4096], X_d [3314,11008]."""
    seed = WORKLOAD_SEED["sweep"]
    return (activations(substream(seed, 0x20), SWEEP_N, 4096),
            activations(substream(seed, 0x21), SWEEP_N, 11008))
