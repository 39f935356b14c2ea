"""q6_K x int8 MMQ prefill GEMM for GB300 (sm_103a): thin Python binding.

Argument marshalling over the C ABI of ``libq6mmq.so`` (declared in
``include/q6mmq.h``): every step of the computation runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There
is no CPU path: calls raise ``Q6Error`` when the library is missing, the
device is not sm_103, or an argument is rejected.
"""
from __future__ import annotations

import ctypes
import dataclasses
import functools
import os
from typing import NamedTuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libq6mmq.so")

Q6_OK, Q6_EINVAL, Q6_EALIGN, Q6_ESIZE, Q6_EARCH, Q6_ECUDA, Q6_ETIMEOUT = range(7)
(PATH_NONE, PATH_TC_RAW, PATH_TC_WEXP, PATH_SKINNY, PATH_TC_WH, PATH_SYNC_WEXP,
 PATH_SKINNY_FUSED, PATH_Q4K_TC_RAW, PATH_Q4K_TC_WQ, PATH_TC_FUSED_RAW,
 PATH_TC_FUSED_WH, PATH_Q4K_SKINNY, PATH_Q4K_SKINNY_FUSED) = range(13)
PATH_NAMES = {PATH_NONE: "none", PATH_TC_RAW: "tc_raw", PATH_TC_WEXP: "tc_wexp",
              PATH_SKINNY: "skinny", PATH_TC_WH: "tc_wh", PATH_SYNC_WEXP: "sync_wexp",
              PATH_SKINNY_FUSED: "skinny_fused", PATH_Q4K_TC_RAW: "q4k_tc_raw",
              PATH_Q4K_TC_WQ: "q4k_tc_wq", PATH_TC_FUSED_RAW: "tc_fused_raw",
              PATH_TC_FUSED_WH: "tc_fused_wh", PATH_Q4K_SKINNY: "q4k_skinny",
              PATH_Q4K_SKINNY_FUSED: "q4k_skinny_fused"}
SKINNY_MAX_N = 16
SKINNY_GROUPS_MAX_N = 96
SKINNY_GROUP_N = 32
Q4K_SKINNY_MAX_N = 16
Q4K_DP4A_MAX_N = 2
Q4K_GROUPS_MAX_N = 64
Q4K_GROUP_N = 32
FUSED_MAX_N = 2

# Every function include/q6mmq.h declares: (name, restype, argtypes).
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
_IP = ctypes.POINTER(ctypes.c_int)
SIGNATURES = [
    ("q6_last_error", ctypes.c_char_p, []),
    ("q6_device_check", _I, []),
    ("q6_sync_status", _I, [_P]),
    ("q6_selftest_wait_timeout", _I, [_I, _P]),
    ("q8_act_plane_bytes", _I, [_I, _I, _SZ, _SZ, _SZ, _IP]),
    ("q8_quantize_act", _I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    ("q6k_plane_bytes", _I, [_I, _I, _SZ, _SZ]),
    ("q6k_pack_weights", _I, [_P, _I, _I, _P, _P, _P, _P]),
    ("q6k_unpack_weights", _I, [_P, _P, _I, _I, _P, _P]),
    ("q6k_mmq_workspace_bytes", _I, [_I, _I, _I, _SZ]),
    ("q6k_tc_part_bytes", _I, [_I, _I, _I, _SZ]),
    ("q6k_mmq_launches", _I, [_I, _I, _I, _I, _IP]),
    ("q6k_mmq", _I, [_P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _P, ctypes.c_size_t, _P, _P,
                     _IP, _P]),
    ("q6k_mmq_noalloc", _I, [_P, _P, _I, _I, _P, _P, _P, _I, _P, _I, _IP, _P]),
    ("q6k_mmq_noalloc_status", _I, [_P]),
    ("q6k_mmq_mma_sync", _I, [_P, _P, _I, _I, _P, _P, _I, _P, _I, _P, _P, _IP, _P]),
    ("q6k_mmq_f32", _I, [_P, _I, _I, _P, _I, _I, _P, _I, _IP, _P]),
    ("q4k_mmq_f32", _I, [_P, _I, _I, _P, _I, _I, _P, _I, _IP, _P]),
    ("q6k_mmq_f32_tc", _I, [_P, _P, _I, _I, _P, _I, _I, _P, _I, _P, ctypes.c_size_t, _IP, _P]),
    ("q8_act_sums_bytes", _I, [_I, _I, _SZ, _IP]),
    ("q8_quantize_act_sums", _I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    ("q4k_plane_bytes", _I, [_I, _I, _SZ, _SZ]),
    ("q4k_pack_weights", _I, [_P, _I, _I, _P, _P, _P]),
    ("q4k_unpack_weights", _I, [_P, _I, _I, _P, _P]),
    ("q4k_mmq", _I, [_P, _P, _I, _I, _P, _P, _P, _P, _I, _P, _I, _P, ctypes.c_size_t, _P, _IP,
                     _P]),
]


class Q6Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"q6mmq error {code}: {msg}")
        self.code = code


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the library (once) and declares every exported signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise Q6Error(-1, f"CUDA library not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != Q6_OK:
        raise Q6Error(rc, load().q6_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _tensor(t, name, dtype, shape, device=None, rows=False):
    """Checks that t is laid out as the C ABI reads it and returns t: a torch
    tensor of this dtype and shape, contiguous (or, with rows=True, a 2-D view
    whose rows are contiguous and do not overlap), on a CUDA device (`device`
    when given). Raises Q6Error(Q6_EINVAL) before anything is launched."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise Q6Error(Q6_EINVAL, f"{name} must be a torch tensor")
    if t.dtype is not dtype:
        raise Q6Error(Q6_EINVAL, f"{name} must be {dtype}, not {t.dtype}")
    if t.shape != shape:
        raise Q6Error(Q6_EINVAL, f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    if not t.is_contiguous() and not (
            rows and t.dim() == 2 and (t.shape[1] <= 1 or t.stride(1) == 1)
            and (t.shape[0] <= 1 or t.stride(0) >= t.shape[1])):
        raise Q6Error(Q6_EINVAL, f"{name} has an unsupported layout (strides {tuple(t.stride())})")
    if not t.is_cuda or (device is not None and t.device != device):
        raise Q6Error(Q6_EINVAL, f"{name} must be a CUDA tensor on {device or 'a CUDA device'}")
    return t


def _same_device(*specs):
    """_tensor() on each (tensor or None, name, dtype, shape), then one CUDA
    device for all of them."""
    devs = {_tensor(t, name, dtype, shape).device for t, name, dtype, shape in specs
            if t is not None}
    if len(devs) > 1:
        raise Q6Error(Q6_EINVAL, f"tensors on different devices: {sorted(map(str, devs))}")


def _row_stride(t):
    """The row stride the C ABI gets for a 2-D rows view (any value >= the
    width is valid; a single row's stride is not used)."""
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------- sizes ---

@functools.lru_cache(maxsize=256)
def act_plane_bytes(N: int, K: int):
    """(xq_bytes, da_bytes, xh_bytes, ldda) of an N x K activation."""
    a, b, c, ld = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    _check(load().q8_act_plane_bytes(N, K, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                     ctypes.byref(ld)))
    return a.value, b.value, c.value, ld.value


@functools.lru_cache(maxsize=256)
def act_sums_bytes(N: int, K: int):
    """(us_bytes, ldus) of the block-sum pairs of an N x K activation."""
    a, ld = ctypes.c_size_t(), ctypes.c_int()
    _check(load().q8_act_sums_bytes(N, K, ctypes.byref(a), ctypes.byref(ld)))
    return a.value, ld.value


@functools.lru_cache(maxsize=256)
def plane_bytes(M: int, K: int):
    """(packed plane bytes, W_exp bytes) of an M x K q6_K weight."""
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().q6k_plane_bytes(M, K, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


# ------------------------------------------------------------ operations ---

@dataclasses.dataclass(frozen=True)
class Activations:
    """Quantised activations on the device: xq [N,K] int8, da [K/32, ldda] f32,
    xh [N,K] f16 (xq or xh may be None), and optionally us [N, ldus] f32, da
    times each 32-block's code sum as hi/lo pairs (the q4_K GEMM's min term
    needs it; see q8_quantize_act_sums in the C header). Checked once, when
    made; read-only."""
    N: int
    K: int
    xq: object
    da: object
    xh: object
    ldda: int
    us: object = None

    def __post_init__(self):
        import torch
        N, K = self.N, self.K
        if self.ldda != act_plane_bytes(N, K)[3]:
            raise Q6Error(Q6_EINVAL, f"ldda {self.ldda} does not match {act_plane_bytes(N, K)[3]}")
        _same_device((self.xq, "xq", torch.int8, (N, K)), (self.xh, "xh", torch.float16, (N, K)),
                     (self.da, "da", torch.float32, (K // 32, self.ldda)),
                     (self.us, "us", torch.float32, (N, act_sums_bytes(N, K)[1])))

    @property
    def device(self):
        return self.da.device


def alloc_activations(N: int, K: int, device=None, want_xh: bool = True,
                      want_xq: bool = True, want_us: bool = False) -> Activations:
    """Buffers for quantised activations. A prefill caller that only runs the
    tensor-core GEMM (N > SKINNY_MAX_N) can skip xq; the few-token kernels
    need it (and not xh), and with xq present and no resident operand plane,
    up to SKINNY_GROUPS_MAX_N (q6_K) or Q4K_GROUPS_MAX_N (q4_K) tokens run
    them on token groups instead of the tensor cores."""
    import torch
    dev = device or torch.device("cuda")
    _, dab, _, ldda = act_plane_bytes(N, K)
    xq = torch.empty((N, K), dtype=torch.int8, device=dev) if want_xq else None
    da = torch.empty((K // 32, ldda), dtype=torch.float32, device=dev)
    xh = torch.empty((N, K), dtype=torch.float16, device=dev) if want_xh else None
    us = (torch.empty((N, act_sums_bytes(N, K)[1]), dtype=torch.float32, device=dev)
          if want_us else None)
    return Activations(N, K, xq, da, xh, ldda, us)


def quantize_act(X, out: Activations | None = None, want_xh: bool = True, stream=None,
                 want_xq: bool = True, want_us: bool = False) -> Activations:
    """Quantises f32 activations X [N, K] (CUDA tensor, last dim contiguous);
    with want_us (or an `out` that has us) also the block sums us."""
    import torch
    if not isinstance(X, torch.Tensor) or X.dim() != 2:
        raise Q6Error(Q6_EINVAL, "X must be a 2-D torch tensor [N, K]")
    N, K = X.shape
    _tensor(X, "X", torch.float32, (N, K), rows=True)
    if out is None:
        out = alloc_activations(N, K, X.device, want_xh, want_xq, want_us)
    elif out.N != N or out.K != K or out.device != X.device:
        raise Q6Error(Q6_EINVAL, f"out holds {out.N} x {out.K} activations on {out.device}, "
                                 f"X is {N} x {K} on {X.device}")
    if out.us is not None:
        _check(load().q8_quantize_act_sums(_ptr(X), N, K, _row_stride(X), _ptr(out.xq),
                                           _ptr(out.da), _ptr(out.xh), _ptr(out.us),
                                           _stream(stream)))
    else:
        _check(load().q8_quantize_act(_ptr(X), N, K, _row_stride(X), _ptr(out.xq),
                                      _ptr(out.da), _ptr(out.xh), _stream(stream)))
    return out


@dataclasses.dataclass(frozen=True)
class Weights:
    """A packed q6_K weight on the device: the packed plane, and optionally the
    W_exp (int8) plane and the resident operand planes wh [2, M, K] binary16
    (W_hi, W_lo: the sub-block scale folded into the centered codes).
    Checked once, when made; read-only."""
    M: int
    K: int
    plane: object
    wexp: object
    wh: object

    def __post_init__(self):
        import torch
        _same_device((self.wexp, "wexp", torch.int8, (self.M, self.K)),
                     (self.wh, "wh", torch.float16, (2, self.M, self.K)),
                     (self.plane, "plane", torch.uint8, (plane_bytes(self.M, self.K)[0],)))

    @property
    def device(self):
        return self.plane.device


def pack_weights(raw, M: int, K: int, wexp: bool = False, wh: bool = False, stream=None,
                 device=None) -> Weights:
    """Packs raw GGUF q6_K bytes: a contiguous uint8 tensor of M*K/256*210
    bytes, on a CUDA device (the planes go there) or in host memory (the
    planes go to `device`, default the current CUDA device). A host tensor is
    page-locked first unless it already is, and the call waits for the pack
    kernel, which reads it directly, before returning."""
    import torch
    pb, wb = plane_bytes(M, K)
    if (not isinstance(raw, torch.Tensor) or raw.numel() != M * (K // 256) * 210
            or raw.dtype != torch.uint8 or not raw.is_contiguous()):
        raise Q6Error(Q6_EINVAL, "raw must be a contiguous uint8 tensor of M*K/256*210 bytes")
    on_host = not raw.is_cuda
    if on_host:
        dev = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        if not raw.is_pinned():
            raw = raw.pin_memory()
    else:
        dev = raw.device
    plane = torch.empty(pb, dtype=torch.uint8, device=dev)
    w8 = torch.empty((M, K), dtype=torch.int8, device=dev) if wexp else None
    w16 = torch.empty((2, M, K), dtype=torch.float16, device=dev) if wh else None
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        _check(load().q6k_pack_weights(_ptr(raw), M, K, _ptr(plane), _ptr(w8), _ptr(w16),
                                       _stream(s)))
        if on_host:
            s.synchronize()      # the kernel has read the host bytes
    return Weights(M, K, plane, w8, w16)


def unpack_weights(w: Weights, out=None, from_wexp: bool = False, stream=None):
    """The weight unpack pass: the binary16 operand planes [2, M, K] (W_hi,
    W_lo) from the packed plane (or from the W_exp plane and the packed
    plane's sub-block scales)."""
    import torch
    dev = w.device
    if out is None:
        out = torch.empty((2, w.M, w.K), dtype=torch.float16, device=dev)
    _tensor(out, "out", torch.float16, (2, w.M, w.K), dev)
    src8 = w.wexp if from_wexp else None
    if from_wexp and src8 is None:
        raise Q6Error(Q6_EINVAL, "weights were packed without the W_exp plane")
    _check(load().q6k_unpack_weights(_ptr(w.plane), _ptr(src8), w.M, w.K, _ptr(out),
                                     _stream(stream)))
    return out


@functools.lru_cache(maxsize=256)
def workspace_bytes(M: int, K: int, N: int) -> int:
    b = ctypes.c_size_t()
    _check(load().q6k_mmq_workspace_bytes(M, K, N, ctypes.byref(b)))
    return b.value


@functools.lru_cache(maxsize=256)
def tc_part_bytes(M: int, K: int, N: int) -> int:
    """Bytes of the K-part partial sums a tensor-core call of this shape uses
    (0 when it does not split K)."""
    b = ctypes.c_size_t()
    _check(load().q6k_tc_part_bytes(M, K, N, ctypes.byref(b)))
    return b.value


def mmq_launches(M: int, K: int, N: int, has_wh: bool) -> int:
    """Kernels one q6k_mmq call launches for this shape on the current device."""
    n = ctypes.c_int()
    _check(load().q6k_mmq_launches(M, K, N, int(bool(has_wh)), ctypes.byref(n)))
    return n.value


class Debug(NamedTuple):
    """The GEMM's optional debug outputs (int32 CUDA tensors, or None):
    partials [N, M, K/16], the exact P = sum over each 16-element sub-block of
    (q - 32) * xq; chunk_sums [N, M, K/32], the exact S = sc[2c] * P[2c] +
    sc[2c+1] * P[2c+1] that the kernel forms per 32-element chunk."""
    partials: object = None
    chunk_sums: object = None


def _debug_buffers(N, M, K, partials, chunk_sums, dev):
    import torch
    if not (partials or chunk_sums):
        return None
    return Debug(
        torch.empty((N, M, K // 16), dtype=torch.int32, device=dev) if partials else None,
        torch.empty((N, M, K // 32), dtype=torch.int32, device=dev) if chunk_sums else None)


_workspaces = {}


def _workspace(nbytes: int, device):
    """A cached device scratch buffer of at least nbytes (one per device)."""
    import torch
    key = str(device)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def mmq(w: Weights, act: Activations, Y=None, source: str = "auto", partials: bool = False,
        workspace=None, wh=None, stream=None, chunk_sums: bool = False):
    """Y [N, M] f32 = the q6_K x int8 GEMM. Returns (Y, path name, Debug or
    None): with partials=True and/or chunk_sums=True the debug outputs (see
    Debug) are filled as well.

    source: "raw" (unpack the packed plane), "wexp" (convert the W_exp plane),
    "wh" (resident binary16 plane) or "auto" (wh, else wexp, else raw). Up to
    SKINNY_MAX_N tokens run the few-token kernels on the packed plane whatever
    the source; when act has xq, up to SKINNY_GROUP_N tokens too whatever the
    source and up to SKINNY_GROUPS_MAX_N when the source is not "wh" (token
    groups of at most SKINNY_GROUP_N)."""
    import torch
    N, M, K = act.N, w.M, w.K
    if act.K != K:
        raise Q6Error(Q6_EINVAL, "activation K does not match the weight")
    if source == "auto":
        source = "wh" if w.wh is not None else ("wexp" if w.wexp is not None else "raw")
    wx = w.wexp if source == "wexp" else None
    w16 = (wh if wh is not None else w.wh) if source == "wh" else None
    if source in ("wexp", "wh") and (wx if source == "wexp" else w16) is None:
        raise Q6Error(Q6_EINVAL, f"weights were packed without the {source} plane")
    dev = w.device
    if wh is not None and w16 is wh:
        _tensor(w16, "wh", torch.float16, (2, M, K), dev)
    if act.device != dev:
        raise Q6Error(Q6_EINVAL, f"activations on {act.device}, weights on {dev}")
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    D = _debug_buffers(N, M, K, partials, chunk_sums, dev)
    ws_need = (workspace_bytes(M, K, N) if (w16 is None or partials)
               else tc_part_bytes(M, K, N) if N > SKINNY_MAX_N else 0)
    if workspace is not None:
        _tensor(workspace, "workspace", getattr(workspace, "dtype", None),
                tuple(getattr(workspace, "shape", ())), dev)
    ws = workspace if workspace is not None else (_workspace(ws_need, dev) if ws_need else None)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    path = ctypes.c_int(-1)
    _check(load().q6k_mmq(_ptr(w.plane), _ptr(wx), _ptr(w16), M, K, _ptr(act.xq), _ptr(act.da),
                          _ptr(act.xh), N, _ptr(Y), _row_stride(Y), _ptr(ws), ws_bytes,
                          _ptr(D and D.partials), _ptr(D and D.chunk_sums), ctypes.byref(path),
                          _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value)), D


def mmq_f32(w: Weights, X, Y=None, stream=None):
    """One or two tokens straight from f32 activations X [N, K] (N <= 2), in
    one kernel: the same Y as quantize_act(X) followed by mmq(). Returns
    (Y, path name)."""
    import torch
    if not isinstance(X, torch.Tensor) or X.dim() != 2:
        raise Q6Error(Q6_EINVAL, "X must be a 2-D torch tensor [N, K]")
    N, K, M = X.shape[0], w.K, w.M
    dev = w.device
    _tensor(X, "X", torch.float32, (N, K), dev, rows=True)
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    path = ctypes.c_int(-1)
    _check(load().q6k_mmq_f32(_ptr(w.plane), M, K, _ptr(X), _row_stride(X), N, _ptr(Y),
                              _row_stride(Y), ctypes.byref(path), _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value))


def mmq_f32_tc(w: Weights, X, Y=None, source: str = "auto", workspace=None, wh=None,
               stream=None):
    """The tensor-core GEMM straight from f32 activations X [N, K], the
    quantiser fused into the GEMM (no Xh or da plane): Y bit for bit that of
    quantize_act(X) followed by mmq() on the tensor-core path. source: "raw"
    (unpack the packed plane), "wh" (resident operand planes) or "auto".
    Returns (Y, path name)."""
    import torch
    if not isinstance(X, torch.Tensor) or X.dim() != 2:
        raise Q6Error(Q6_EINVAL, "X must be a 2-D torch tensor [N, K]")
    N, K, M = X.shape[0], w.K, w.M
    dev = w.device
    _tensor(X, "X", torch.float32, (N, K), dev, rows=True)
    if source == "auto":
        source = "wh" if (wh is not None or w.wh is not None) else "raw"
    if source not in ("raw", "wh"):
        raise Q6Error(Q6_EINVAL, f"source must be raw, wh or auto, not {source}")
    w16 = (wh if wh is not None else w.wh) if source == "wh" else None
    if source == "wh" and w16 is None:
        raise Q6Error(Q6_EINVAL, "weights were packed without the wh plane")
    if w16 is not None:
        _tensor(w16, "wh", torch.float16, (2, M, K), dev)
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    part = tc_part_bytes(M, K, N)
    ws_need = (-(-4 * M * K // 256) * 256 + part) if w16 is None else part
    if workspace is not None:
        _tensor(workspace, "workspace", getattr(workspace, "dtype", None),
                tuple(getattr(workspace, "shape", ())), dev)
    ws = workspace if workspace is not None else (_workspace(ws_need, dev) if ws_need else None)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    path = ctypes.c_int(-1)
    _check(load().q6k_mmq_f32_tc(_ptr(w.plane), _ptr(w16), M, K, _ptr(X), _row_stride(X), N,
                                 _ptr(Y), _row_stride(Y), _ptr(ws), ws_bytes, ctypes.byref(path),
                                 _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value))


def mmq_mma_sync(w: Weights, act: Activations, Y=None, partials: bool = False, stream=None,
                 chunk_sums: bool = False):
    """The same GEMM on the legacy mma.sync int8 path (the pages' route), from
    the W_exp plane: a comparison point for mmq(). Returns (Y, path, Debug or
    None)."""
    import torch
    N, M, K = act.N, w.M, w.K
    if act.K != K:
        raise Q6Error(Q6_EINVAL, "activation K does not match the weight")
    if w.wexp is None:
        raise Q6Error(Q6_EINVAL, "weights were packed without the wexp plane")
    dev = w.device
    if act.device != dev:
        raise Q6Error(Q6_EINVAL, f"activations on {act.device}, weights on {dev}")
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    D = _debug_buffers(N, M, K, partials, chunk_sums, dev)
    path = ctypes.c_int(-1)
    _check(load().q6k_mmq_mma_sync(_ptr(w.plane), _ptr(w.wexp), M, K, _ptr(act.xq), _ptr(act.da), N,
                                   _ptr(Y), _row_stride(Y), _ptr(D and D.partials),
                                   _ptr(D and D.chunk_sums), ctypes.byref(path), _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value)), D


def sync_status(stream=None):
    """Waits for the stream and raises if a kernel gave up a bounded wait."""
    _check(load().q6_sync_status(_stream(stream)))


# ------------------------------------------------------------------- q4_K ---

@functools.lru_cache(maxsize=256)
def q4k_plane_bytes(M: int, K: int):
    """(packed q4_K plane bytes, operand plane bytes) of an M x K weight."""
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().q4k_plane_bytes(M, K, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


@dataclasses.dataclass(frozen=True)
class Q4Weights:
    """A packed q4_K weight on the device: the packed plane and optionally the
    resident binary16 operand plane wq [M, K] (sc * q). Checked once, when
    made; read-only."""
    M: int
    K: int
    plane: object
    wq: object

    def __post_init__(self):
        import torch
        _same_device((self.wq, "wq", torch.float16, (self.M, self.K)),
                     (self.plane, "plane", torch.uint8, (q4k_plane_bytes(self.M, self.K)[0],)))

    @property
    def device(self):
        return self.plane.device


def q4k_pack_weights(raw, M: int, K: int, wq: bool = False, stream=None,
                     device=None) -> Q4Weights:
    """Packs raw GGUF q4_K bytes (a contiguous uint8 tensor of M*K/256*144
    bytes, on a CUDA device or in host memory, as pack_weights)."""
    import torch
    pb, wb = q4k_plane_bytes(M, K)
    if (not isinstance(raw, torch.Tensor) or raw.numel() != M * (K // 256) * 144
            or raw.dtype != torch.uint8 or not raw.is_contiguous()):
        raise Q6Error(Q6_EINVAL, "raw must be a contiguous uint8 tensor of M*K/256*144 bytes")
    on_host = not raw.is_cuda
    if on_host:
        dev = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        if not raw.is_pinned():
            raw = raw.pin_memory()
    else:
        dev = raw.device
    plane = torch.empty(pb, dtype=torch.uint8, device=dev)
    w16 = torch.empty((M, K), dtype=torch.float16, device=dev) if wq else None
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        _check(load().q4k_pack_weights(_ptr(raw), M, K, _ptr(plane), _ptr(w16), _stream(s)))
        if on_host:
            s.synchronize()
    return Q4Weights(M, K, plane, w16)


def q4k_unpack_weights(w: Q4Weights, out=None, stream=None):
    """The q4_K unpack pass: the binary16 operand plane [M, K] = sc * q."""
    import torch
    if out is None:
        out = torch.empty((w.M, w.K), dtype=torch.float16, device=w.device)
    _tensor(out, "out", torch.float16, (w.M, w.K), w.device)
    _check(load().q4k_unpack_weights(_ptr(w.plane), w.M, w.K, _ptr(out), _stream(stream)))
    return out


def q4k_mmq_f32(w: Q4Weights, X, Y=None, stream=None):
    """One or two tokens of the q4_K GEMM straight from f32 activations X
    [N, K] (N <= 2), in one kernel: the same Y, bit for bit, as
    quantize_act(X, want_us=True) followed by q4k_mmq(). Returns (Y, path
    name)."""
    import torch
    if not isinstance(X, torch.Tensor) or X.dim() != 2:
        raise Q6Error(Q6_EINVAL, "X must be a 2-D torch tensor [N, K]")
    N, K, M = X.shape[0], w.K, w.M
    dev = w.device
    _tensor(X, "X", torch.float32, (N, K), dev, rows=True)
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    path = ctypes.c_int(-1)
    _check(load().q4k_mmq_f32(_ptr(w.plane), M, K, _ptr(X), _row_stride(X), N, _ptr(Y),
                              _row_stride(Y), ctypes.byref(path), _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value))


def q4k_mmq(w: Q4Weights, act: Activations, Y=None, source: str = "auto",
            partials: bool = False, workspace=None, stream=None):
    """Y [N, M] f32 = the q4_K x int8 GEMM. act needs da and us
    (quantize_act(..., want_us=True)), and xq for N <= Q4K_SKINNY_MAX_N (the
    few-token kernels on the packed plane) or xh for more tokens (the tensor
    cores; when xq is there, up to Q4K_GROUP_N tokens on either source and
    up to Q4K_GROUPS_MAX_N from the packed plane run the few-token kernel on
    token groups of at most Q4K_GROUP_N). source (tensor
    cores): "raw" (unpack the packed plane per call), "wq" (the resident
    operand plane) or "auto". Returns (Y, path name, partials [N, M, K/32]
    int32 or None)."""
    import torch
    N, M, K = act.N, w.M, w.K
    if act.K != K:
        raise Q6Error(Q6_EINVAL, "activation K does not match the weight")
    skinny = N <= Q4K_SKINNY_MAX_N
    if source == "auto":
        source = "wq" if w.wq is not None else "raw"
    if source == "wq" and w.wq is None:
        raise Q6Error(Q6_EINVAL, "weights were packed without the wq plane")
    wq = w.wq if source == "wq" else None
    groups = (not skinny and act.xq is not None
              and (N <= Q4K_GROUP_N or (N <= Q4K_GROUPS_MAX_N and wq is None)))
    if (act.us is None or (skinny and act.xq is None)
            or (not skinny and not groups and act.xh is None)):
        raise Q6Error(Q6_EINVAL, "the q4_K GEMM needs activations with us, and xq for "
                                 f"N <= {Q4K_SKINNY_MAX_N} or xh for more tokens")
    skinny = skinny or groups
    dev = w.device
    if act.device != dev:
        raise Q6Error(Q6_EINVAL, f"activations on {act.device}, weights on {dev}")
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=dev)
    _tensor(Y, "Y", torch.float32, (N, M), dev, rows=True)
    P = torch.empty((N, M, K // 32), dtype=torch.int32, device=dev) if partials else None
    part = tc_part_bytes(M, K, N) if not skinny else 0
    need = ((-(-2 * M * K // 256) * 256 + part) if (not skinny and (wq is None or partials))
            else part)
    if workspace is not None:
        _tensor(workspace, "workspace", getattr(workspace, "dtype", None),
                tuple(getattr(workspace, "shape", ())), dev)
    ws = workspace if workspace is not None else (_workspace(need, dev) if need else None)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    path = ctypes.c_int(-1)
    _check(load().q4k_mmq(_ptr(w.plane), _ptr(wq), M, K, _ptr(act.xq), _ptr(act.xh),
                          _ptr(act.da), _ptr(act.us), N, _ptr(Y), _row_stride(Y), _ptr(ws),
                          ws_bytes, _ptr(P), ctypes.byref(path), _stream(stream)))
    return Y, PATH_NAMES.get(path.value, str(path.value)), P
