"""The C-ABI library builds, loads and exports what include/q6mmq.h declares (CPU only).

Only host-side argument checks are called here: every such call returns before
touching a device, so no GPU is needed.
"""
import ctypes
import os
import re

import pytest

import q6_int8_mmq_gb300 as q6
from q6_int8_mmq_gb300 import build as q6build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q6mmq.h")


@pytest.fixture(scope="module")
def lib():
    q6build.build()
    return q6.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(q[68]\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q8_quantize_act", "q6k_pack_weights", "q6k_mmq", "q8_act_plane_bytes",
                     "q6k_plane_bytes", "q6_last_error", "q6_sync_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    bound = {name for name, _, _ in q6.SIGNATURES}
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
        assert name in bound, f"{name} has no binding"


def test_plane_sizes(lib):
    pb, wb = q6.plane_bytes(4096, 11008)
    M, K = 4096, 11008
    r = lambda x: (x + 255) // 256 * 256
    ldm = (M + 3) // 4 * 4
    d_row = (K // 256 * 2 + 15) // 16 * 16
    assert pb == r(M * K * 3 // 4) + r(M * K // 16) + r(M * d_row) + r(K // 256 * ldm * 4)
    assert wb == M * K
    xq, dab, xh, ldda = q6.act_plane_bytes(3314, 11008)
    assert (xq, xh, ldda) == (3314 * 11008, 3314 * 11008 * 2, 3316)
    assert dab == 11008 // 32 * 3316 * 4
    # the q4_K block-sum pairs: 16 values per super-block, an even count of them
    assert q6.act_sums_bytes(3314, 11008) == (3314 * 704 * 4, 704)
    assert q6.act_sums_bytes(5, 512) == (5 * 32 * 4, 32)
    assert q6.act_sums_bytes(5, 256) == (5 * 32 * 4, 32)


@pytest.mark.parametrize("M,K", [(0, 256), (4, 0), (4, 100), (4, 255), (-1, 256)])
def test_plane_bytes_rejects(lib, M, K):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.q6k_plane_bytes(M, K, ctypes.byref(a), ctypes.byref(b)) == q6.Q6_EINVAL
    assert lib.q6_last_error()


def test_host_side_rejections(lib):
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: rejected before any use
    odd = ctypes.c_void_p(0x10004)
    path = ctypes.c_int(-1)

    # N = 97: past the token groups, so the tensor-core path's checks apply
    def mmq(plane=fake, wexp=None, wh=None, M=64, K=256, xq=fake, da=fake, xh=fake, N=97,
            Y=fake, ldy=64, ws=fake, ws_bytes=1 << 30, partials=None, chunk_sums=None):
        return lib.q6k_mmq(plane, wexp, wh, M, K, xq, da, xh, N, Y, ldy, ws, ws_bytes, partials,
                           chunk_sums, ctypes.byref(path), None)

    assert mmq(K=300) == q6.Q6_EINVAL                       # K not a multiple of 256
    assert path.value == q6.PATH_NONE
    assert mmq(ldy=32) == q6.Q6_EINVAL                      # ldy < M
    assert mmq(N=0, xq=None, da=None, xh=None) == q6.Q6_OK  # empty: a no-op
    assert path.value == q6.PATH_NONE
    assert mmq(xh=None) == q6.Q6_EINVAL                     # operand plane needed for N > 96
    assert mmq(N=40, xq=None, xh=None) == q6.Q6_EINVAL      # ... and for N > 16 without Xq
    assert mmq(N=40, wh=fake, xh=None) == q6.Q6_EINVAL      # ... or with resident planes
    assert mmq(N=8, xq=None) == q6.Q6_EINVAL                # int8 activations needed for N <= 16
    assert mmq(da=odd) == q6.Q6_EALIGN                      # misaligned da
    assert mmq(ws=odd) == q6.Q6_EALIGN                      # misaligned workspace
    assert mmq(ws=None) == q6.Q6_ESIZE                      # unpack needs a workspace
    assert mmq(ws_bytes=64 * 256 * 4 - 1) == q6.Q6_ESIZE    # ... of M*K*4 bytes
    # resident planes need no workspace, unless the sub-block partials are wanted
    assert mmq(wh=fake, ws=None, partials=fake) == q6.Q6_ESIZE
    odd1 = ctypes.c_void_p(0x10001)                           # not 4-byte aligned
    assert mmq(partials=odd1) == q6.Q6_EALIGN               # misaligned debug outputs
    assert mmq(chunk_sums=odd1) == q6.Q6_EALIGN
    assert lib.q6k_mmq_mma_sync(fake, fake, 64, 256, fake, fake, 8, fake, 64, None, odd1,
                                ctypes.byref(path), None) == q6.Q6_EALIGN
    size = ctypes.c_size_t()
    assert lib.q6k_mmq_workspace_bytes(64, 256, 64, ctypes.byref(size)) == q6.Q6_OK
    assert size.value == 64 * 256 * 4
    assert lib.q6k_mmq_workspace_bytes(64, 256, 16, ctypes.byref(size)) == q6.Q6_OK
    assert size.value == 0
    # quantiser: ldx < K, misaligned X, N == 0
    assert lib.q8_quantize_act(fake, 4, 256, 128, fake, fake, None, None) == q6.Q6_EINVAL
    assert lib.q8_quantize_act(odd, 4, 256, 256, fake, fake, None, None) == q6.Q6_EALIGN
    assert lib.q8_quantize_act(None, 0, 256, 256, None, None, None, None) == q6.Q6_OK
    # quantiser: neither Xq nor Xh; a misaligned Xq or Xh
    assert lib.q8_quantize_act(fake, 4, 256, 256, None, fake, None, None) == q6.Q6_EINVAL
    assert lib.q8_quantize_act(fake, 4, 256, 256, odd, fake, None, None) == q6.Q6_EALIGN
    assert lib.q8_quantize_act(fake, 4, 256, 256, None, fake, odd, None) == q6.Q6_EALIGN
    # pack: misaligned plane or wh, missing raw
    assert lib.q6k_pack_weights(fake, 4, 256, odd, None, None, None) == q6.Q6_EALIGN
    assert lib.q6k_pack_weights(fake, 4, 256, fake, None, odd, None) == q6.Q6_EALIGN
    assert lib.q6k_pack_weights(None, 4, 256, fake, None, None, None) == q6.Q6_EINVAL
    assert lib.q6_selftest_wait_timeout(0, None) == q6.Q6_EINVAL
    # fused one/two-token call: too many tokens, ldx < K, ldy < M, misaligned X
    # or ldx, K beyond the shared-memory staging, the empty case
    def f32(plane=fake, M=64, K=256, X=fake, ldx=256, N=1, Y=fake, ldy=64):
        return lib.q6k_mmq_f32(plane, M, K, X, ldx, N, Y, ldy, ctypes.byref(path), None)

    assert f32(N=3) == q6.Q6_EINVAL and path.value == q6.PATH_NONE
    assert f32(ldx=128) == q6.Q6_EINVAL
    assert f32(ldy=32) == q6.Q6_EINVAL
    assert f32(X=None) == q6.Q6_EINVAL
    assert f32(X=odd) == q6.Q6_EALIGN
    assert f32(ldx=258) == q6.Q6_EALIGN                    # ldx % 4 != 0
    assert f32(plane=odd) == q6.Q6_EALIGN
    assert f32(K=103168 + 256, ldx=103424, N=2) == q6.Q6_ESIZE
    assert f32(K=206592 + 256, ldx=206848, N=1) == q6.Q6_ESIZE
    assert f32(N=0, X=None, Y=None) == q6.Q6_OK and path.value == q6.PATH_NONE

    # the tensor-core GEMM with the fused quantiser: ldx < K, ldy < M, misaligned
    # X / ldx / wh / workspace, no workspace for the unpack, the empty case
    def f32tc(plane=fake, wh=fake, M=64, K=256, X=fake, ldx=256, N=64, Y=fake, ldy=64,
              ws=None, ws_bytes=0):
        return lib.q6k_mmq_f32_tc(plane, wh, M, K, X, ldx, N, Y, ldy, ws, ws_bytes,
                                  ctypes.byref(path), None)

    assert f32tc(ldx=128) == q6.Q6_EINVAL and path.value == q6.PATH_NONE
    assert f32tc(ldy=32) == q6.Q6_EINVAL
    assert f32tc(X=None) == q6.Q6_EINVAL
    assert f32tc(K=100, ldx=100) == q6.Q6_EINVAL
    assert f32tc(X=odd) == q6.Q6_EALIGN
    assert f32tc(ldx=258) == q6.Q6_EALIGN
    assert f32tc(wh=odd) == q6.Q6_EALIGN
    assert f32tc(plane=odd) == q6.Q6_EALIGN
    assert f32tc(wh=None) == q6.Q6_ESIZE                   # the unpack needs a workspace
    assert f32tc(wh=None, ws=fake, ws_bytes=64 * 256 * 4 - 1) == q6.Q6_ESIZE
    assert f32tc(N=0, X=None, Y=None) == q6.Q6_OK and path.value == q6.PATH_NONE

    # the fused one/two-token q4_K call: N <= 2, ldx, alignment, the shared-memory
    # limit on K, the empty case
    def q4f(plane=fake, M=64, K=256, X=fake, ldx=256, N=1, Y=fake, ldy=64):
        return lib.q4k_mmq_f32(plane, M, K, X, ldx, N, Y, ldy, ctypes.byref(path), None)

    assert q4f(N=3) == q6.Q6_EINVAL and path.value == q6.PATH_NONE
    assert q4f(ldx=128) == q6.Q6_EINVAL
    assert q4f(X=None) == q6.Q6_EINVAL
    assert q4f(X=odd) == q6.Q6_EALIGN
    assert q4f(ldx=258) == q6.Q6_EALIGN
    assert q4f(plane=odd) == q6.Q6_EALIGN
    assert q4f(K=92928 + 256, ldx=92928 + 256, N=2) == q6.Q6_ESIZE
    assert q4f(K=185856 + 256, ldx=185856 + 256, N=1) == q6.Q6_ESIZE
    assert q4f(N=0, X=None, Y=None) == q6.Q6_OK and path.value == q6.PATH_NONE

    # the q4_K GEMM: Xq for N <= 16; Xh beyond, unless Xq is there and N <= 32,
    # or the plane is not resident and N <= 64 (token groups); ldy < M, K % 256,
    # misaligned pointers, no workspace for the tensor-core unpack, the empty
    # case (every call here is refused on the host before any launch)
    def q4(plane=fake, wq=None, M=64, K=256, Xq=fake, Xh=fake, da=fake, us=fake, N=4, Y=fake,
           ldy=64, ws=None, ws_bytes=0, P=None):
        return lib.q4k_mmq(plane, wq, M, K, Xq, Xh, da, us, N, Y, ldy, ws, ws_bytes, P,
                           ctypes.byref(path), None)

    assert q4(Xq=None) == q6.Q6_EINVAL and path.value == q6.PATH_NONE
    assert q4(N=65, Xh=None) == q6.Q6_EINVAL
    assert q4(N=20, Xq=None, Xh=None) == q6.Q6_EINVAL
    assert q4(N=33, wq=fake, Xh=None) == q6.Q6_EINVAL     # past 32, groups only from the packed plane
    assert q4(us=None) == q6.Q6_EINVAL
    assert q4(ldy=32) == q6.Q6_EINVAL
    assert q4(K=300) == q6.Q6_EINVAL
    assert q4(Xq=odd) == q6.Q6_EALIGN
    assert q4(us=odd) == q6.Q6_EALIGN
    assert q4(plane=odd) == q6.Q6_EALIGN
    assert q4(P=odd1) == q6.Q6_EALIGN
    assert q4(N=65) == q6.Q6_ESIZE                         # no workspace for the unpack
    assert q4(N=20, Xq=None) == q6.Q6_ESIZE
    assert q4(N=0, Xq=None, Xh=None, Y=None) == q6.Q6_OK and path.value == q6.PATH_NONE


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(q6.Q6Error):
        q6.load(str(tmp_path / "nope.so"))


def test_binding_checks_tensor_layouts():
    """The binding refuses a tensor the C ABI would misread (wrong dtype,
    shape, overlapping or non-contiguous rows, host memory) before anything is
    launched; a rows view with a wider row stride is accepted as it is."""
    import numpy as np
    import torch
    t = torch.zeros(4, 8)
    with pytest.raises(q6.Q6Error, match="float16"):
        q6._tensor(t, "Y", torch.float16, (4, 8))
    with pytest.raises(q6.Q6Error, match="shape"):
        q6._tensor(t, "Y", torch.float32, (4, 7))
    with pytest.raises(q6.Q6Error, match="torch tensor"):
        q6._tensor(np.zeros((4, 8), np.float32), "Y", torch.float32, (4, 8))
    with pytest.raises(q6.Q6Error, match="layout"):          # columns not contiguous
        q6._tensor(torch.zeros(8, 4).t(), "Y", torch.float32, (4, 8), rows=True)
    with pytest.raises(q6.Q6Error, match="layout"):          # rows overlap
        q6._tensor(torch.zeros(40).as_strided((4, 8), (5, 1)), "Y", torch.float32, (4, 8),
                   rows=True)
    wide = torch.zeros(4, 13)[:, :8]
    with pytest.raises(q6.Q6Error, match="layout"):          # contiguity required
        q6._tensor(wide, "xq", torch.float32, (4, 8))
    with pytest.raises(q6.Q6Error, match="CUDA"):            # layout fine, host memory
        q6._tensor(wide, "Y", torch.float32, (4, 8), rows=True)
    assert q6._row_stride(wide) == 13
    assert q6._row_stride(torch.zeros(1, 8)) == 8
    assert q6._row_stride(torch.zeros(0, 8)) == 8


def test_quantize_refuses_bad_inputs_on_the_host():
    import torch
    with pytest.raises(q6.Q6Error, match="float32"):
        q6.quantize_act(torch.zeros(2, 256, dtype=torch.float64))
    with pytest.raises(q6.Q6Error, match="layout"):
        q6.quantize_act(torch.zeros(256, 2).t())
    with pytest.raises(q6.Q6Error, match="2-D"):
        q6.quantize_act(torch.zeros(256))
    with pytest.raises(q6.Q6Error, match="CUDA"):
        q6.quantize_act(torch.zeros(2, 256))


def test_binding_objects_are_checked_when_made():
    """Activations and Weights validate their tensors once, when made (the
    per-call work is then only the caller's own buffers)."""
    import torch
    ldda = q6.act_plane_bytes(4, 256)[3]
    with pytest.raises(q6.Q6Error, match="ldda"):
        q6.Activations(4, 256, None, torch.zeros(8, ldda), None, ldda + 4)
    with pytest.raises(q6.Q6Error, match="shape"):
        q6.Activations(4, 256, None, torch.zeros(8, ldda + 1), None, ldda)
    with pytest.raises(q6.Q6Error, match="int8"):
        q6.Activations(4, 256, torch.zeros(4, 256), torch.zeros(8, ldda), None, ldda)
    with pytest.raises(q6.Q6Error, match="CUDA"):
        q6.Activations(4, 256, None, torch.zeros(8, ldda), None, ldda)
    pb = q6.plane_bytes(128, 256)[0]
    with pytest.raises(q6.Q6Error, match="shape"):
        q6.Weights(128, 256, torch.zeros(pb - 1, dtype=torch.uint8), None, None)
    with pytest.raises(q6.Q6Error, match="CUDA"):
        q6.Weights(128, 256, torch.zeros(pb, dtype=torch.uint8), None, None)


def test_binding_constants_match_the_header():
    """The routing limits the binding mirrors (token counts of the few-token
    paths, the token groups, the fused calls) equal the header's #defines, so
    the binding sizes its buffers for the path the library takes."""
    text = open(HEADER).read()
    defines = {k: int(v) for k, v in re.findall(r"^#define\s+Q6_(\w+)\s+(\d+)", text, flags=re.M)}
    for name in ("SKINNY_MAX_N", "SKINNY_GROUPS_MAX_N", "SKINNY_GROUP_N", "FUSED_MAX_N",
                 "Q4K_SKINNY_MAX_N", "Q4K_DP4A_MAX_N", "Q4K_GROUPS_MAX_N", "Q4K_GROUP_N"):
        assert getattr(q6, name) == defines[name], name
    assert q6.SKINNY_GROUP_N >= q6.SKINNY_MAX_N and q6.Q4K_GROUP_N >= q6.Q4K_SKINNY_MAX_N
