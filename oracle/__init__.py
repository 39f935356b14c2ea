"""CPU oracle for the q6_K x int8 GEMM -- TEST INFRASTRUCTURE ONLY.

Loads ``q6k_oracle.c`` and ``q4k_oracle.c`` (plain single-threaded C, built
with gcc into one shared object) through ctypes. Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package; the CUDA library never does.
The C source cites the passages of the pages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q6k_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "q4k_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fexcess-precision=standard",
          "-fPIC", "-shared", "-Wall"]


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    name = "liborc.so" if mutant == 0 else f"liborc_m{mutant}.so"
    out = os.path.join(_BUILD, name)
    if force or not os.path.exists(out) or any(
            os.path.getmtime(out) < os.path.getmtime(src) for src in _SRCS):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, f"-DORC_MUTANT={mutant}", "-o", tmp, *_SRCS, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I = ctypes.c_int


class Oracle:
    """ctypes front of one build of the oracle."""

    def __init__(self, mutant: int = 0):
        self.path = build(mutant)
        lib = ctypes.CDLL(self.path)
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_q6k_decode_block.argtypes = [_P, _P]
        lib.orc_q6k_wexp.argtypes = [_P, _I, _I, _P]
        lib.orc_q6k_dsc.argtypes = [_P, _I, _I, _P]
        lib.orc_q8_quantize.argtypes = [_P, _I, _I, _I, _P, _P]
        lib.orc_mmq.argtypes = [_P, _I, _I, _P, _P, _I, _P, _P]
        lib.orc_mutant.restype = _I
        lib.orc_q4k_scale_min.argtypes = [_P, _I, _P, _P]
        lib.orc_q4k_decode_block.argtypes = [_P, _P, _P, _P, _P, _P]
        lib.orc_q4k_mmq.argtypes = [_P, _I, _I, _P, _P, _I, _P, _P]
        self.lib = lib
        self.mutant = lib.orc_mutant()

    @staticmethod
    def _ptr(a: np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data_as(ctypes.c_void_p)

    def f16_to_f64(self, h: int) -> float:
        return self.lib.orc_f16_to_f64(int(h) & 0xFFFF)

    def decode_block(self, blk: np.ndarray) -> np.ndarray:
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        assert blk.size == 210
        out = np.empty(256, dtype=np.int8)
        self.lib.orc_q6k_decode_block(self._ptr(blk), self._ptr(out))
        return out

    def wexp(self, raw: np.ndarray, M: int, K: int) -> np.ndarray:
        raw = np.ascontiguousarray(raw, dtype=np.uint8)
        assert raw.size == M * (K // 256) * 210
        out = np.empty((M, K), dtype=np.int8)
        self.lib.orc_q6k_wexp(self._ptr(raw), M, K, self._ptr(out))
        return out

    def dsc(self, raw: np.ndarray, M: int, K: int) -> np.ndarray:
        raw = np.ascontiguousarray(raw, dtype=np.uint8)
        assert raw.size == M * (K // 256) * 210
        out = np.empty((M, K // 16), dtype=np.float32)
        self.lib.orc_q6k_dsc(self._ptr(raw), M, K, self._ptr(out))
        return out

    def quantize(self, X: np.ndarray):
        """(xq int8 [N,K], da f32 [N,K/32])."""
        X = np.ascontiguousarray(X, dtype=np.float32)
        N, K = X.shape
        assert K % 32 == 0
        xq = np.empty((N, K), dtype=np.int8)
        da = np.empty((N, K // 32), dtype=np.float32)
        self.lib.orc_q8_quantize(self._ptr(X), N, K, K, self._ptr(xq), self._ptr(da))
        return xq, da

    def mmq(self, raw: np.ndarray, M: int, K: int, xq: np.ndarray, da: np.ndarray,
            partials: bool = False):
        """Y f64 [N,M] (and int32 partials [N,M,K/16] when asked)."""
        raw = np.ascontiguousarray(raw, dtype=np.uint8)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        da = np.ascontiguousarray(da, dtype=np.float32)
        N = xq.shape[0]
        assert raw.size == M * (K // 256) * 210 and xq.shape == (N, K)
        assert da.shape == (N, K // 32)
        Y = np.empty((N, M), dtype=np.float64)
        P = np.empty((N, M, K // 16), dtype=np.int32) if partials else None
        self.lib.orc_mmq(self._ptr(raw), M, K, self._ptr(xq), self._ptr(da), N,
                         self._ptr(Y), self._ptr(P) if partials else None)
        return (Y, P) if partials else Y


    def mmq_all(self, raw: np.ndarray, M: int, K: int, xq: np.ndarray, da: np.ndarray,
                threads: int | None = None) -> np.ndarray:
        """Y f64 [N,M] for large shapes: the same orc_mmq run on disjoint ranges
        of weight rows from several threads (ctypes releases the GIL), so every
        output element comes from the unchanged single-threaded loop."""
        import concurrent.futures as cf
        raw = np.ascontiguousarray(raw, dtype=np.uint8).reshape(M, -1)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        da = np.ascontiguousarray(da, dtype=np.float32)
        N = xq.shape[0]
        T = max(1, min(threads or os.cpu_count() or 1, M))
        bounds = [M * i // T for i in range(T + 1)]
        parts = [None] * T

        def run(i):
            m0, m1 = bounds[i], bounds[i + 1]
            sub = np.ascontiguousarray(raw[m0:m1])
            y = np.empty((N, m1 - m0), dtype=np.float64)
            self.lib.orc_mmq(self._ptr(sub), m1 - m0, K, self._ptr(xq), self._ptr(da), N,
                             self._ptr(y), None)
            parts[i] = y

        with cf.ThreadPoolExecutor(max_workers=T) as ex:
            list(ex.map(run, range(T)))
        return np.concatenate(parts, axis=1)


    # ------------------------------------------------------------- q4_K --

    def q4k_scale_min(self, s12: np.ndarray, j: int):
        """(scale, min) of sub-block j from the 12 packed bytes."""
        s12 = np.ascontiguousarray(s12, dtype=np.uint8)
        assert s12.size == 12
        sc, mn = ctypes.c_int(), ctypes.c_int()
        self.lib.orc_q4k_scale_min(self._ptr(s12), j, ctypes.byref(sc), ctypes.byref(mn))
        return sc.value, mn.value

    def q4k_decode_block(self, blk: np.ndarray):
        """(codes uint8 [256], sc int [8], mins int [8], d, dmin) of one block."""
        blk = np.ascontiguousarray(blk, dtype=np.uint8)
        assert blk.size == 144
        codes = np.empty(256, np.uint8)
        sc = np.empty(8, np.intc)
        mn = np.empty(8, np.intc)
        d, dmin = ctypes.c_double(), ctypes.c_double()
        self.lib.orc_q4k_decode_block(self._ptr(blk), self._ptr(codes), self._ptr(sc),
                                      self._ptr(mn), ctypes.byref(d), ctypes.byref(dmin))
        return codes, sc.astype(np.int64), mn.astype(np.int64), d.value, dmin.value

    def q4k_mmq(self, raw: np.ndarray, M: int, K: int, xq: np.ndarray, da: np.ndarray,
                partials: bool = False):
        """Y f64 [N,M] of the q4_K GEMM (and int32 partials [N,M,K/32] when asked)."""
        raw = np.ascontiguousarray(raw, dtype=np.uint8)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        da = np.ascontiguousarray(da, dtype=np.float32)
        N = xq.shape[0]
        assert raw.size == M * (K // 256) * 144 and xq.shape == (N, K)
        assert da.shape == (N, K // 32)
        Y = np.empty((N, M), dtype=np.float64)
        P = np.empty((N, M, K // 32), dtype=np.int32) if partials else None
        self.lib.orc_q4k_mmq(self._ptr(raw), M, K, self._ptr(xq), self._ptr(da), N,
                             self._ptr(Y), self._ptr(P) if partials else None)
        return (Y, P) if partials else Y

    def q4k_mmq_all(self, raw: np.ndarray, M: int, K: int, xq: np.ndarray, da: np.ndarray,
                    threads: int | None = None) -> np.ndarray:
        """q4k_mmq over disjoint weight-row ranges from several threads (every
        output element from the unchanged single-threaded loop)."""
        import concurrent.futures as cf
        raw = np.ascontiguousarray(raw, dtype=np.uint8).reshape(M, -1)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        da = np.ascontiguousarray(da, dtype=np.float32)
        N = xq.shape[0]
        T = max(1, min(threads or os.cpu_count() or 1, M))
        bounds = [M * i // T for i in range(T + 1)]
        parts = [None] * T

        def run(i):
            m0, m1 = bounds[i], bounds[i + 1]
            sub = np.ascontiguousarray(raw[m0:m1])
            y = np.empty((N, m1 - m0), dtype=np.float64)
            self.lib.orc_q4k_mmq(self._ptr(sub), m1 - m0, K, self._ptr(xq), self._ptr(da), N,
                                 self._ptr(y), None)
            parts[i] = y

        with cf.ThreadPoolExecutor(max_workers=T) as ex:
            list(ex.map(run, range(T)))
        return np.concatenate(parts, axis=1)


_default = None


def get() -> Oracle:
    """The (lazily built) default oracle."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
