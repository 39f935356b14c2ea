"""Parity of the CUDA library with the CPU oracle (needs a GB300).

Integer results (quantised activations, packed planes, the debug partials)
must be bit-exact. The kernels have two debug outputs: the sub-block partials
P[n][m][s] = sum over the 16 elements of sub-block s of (q - 32) * xq, which
are compared with the oracle's P directly, and the chunk sums the kernels form
themselves, S[n][m][c] = sc[m][2c] * P[2c] + sc[m][2c+1] * P[2c+1], whose
expected value is formed here from the oracle's P and the raw sub-block
scales. Y must satisfy the floating-point tolerance of the method:
max|Y - Yo| <= 1e-3 * max|Yo| and sum|Y - Yo| / sum|Yo| <= 1e-5 (the normwise
reading of "mean relative error"). Full-size workloads are checked on every
output, in the launch configuration the benchmark uses, against the oracle run
over disjoint weight-row ranges on the host cores; their debug partials are
checked bit-exactly on sampled tokens.
"""
import ctypes
import dataclasses

import numpy as np
import pytest

import oracle
import restate
from q6_int8_mmq_gb300 import synth

pytestmark = pytest.mark.gpu

MAX_REL = 1e-3
NORMWISE = 1e-5


@pytest.fixture(scope="module")
def q6():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q6_int8_mmq_gb300 as q6mod
    from q6_int8_mmq_gb300 import build as q6build
    q6build.build()
    q6mod.load()
    return q6mod


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def check_y(Y, Yo, label=""):
    Y = np.asarray(Y, dtype=np.float64)
    err = np.abs(Y - Yo)
    scale = np.abs(Yo).max()
    assert np.all(np.isfinite(Y)), label
    if scale == 0:
        assert err.max() == 0, label
        return
    maxrel = err.max() / scale
    normwise = err.sum() / np.abs(Yo).sum()
    assert maxrel <= MAX_REL, f"{label}: max error {maxrel:.3e} of max|Y|"
    assert normwise <= NORMWISE, f"{label}: normwise error {normwise:.3e}"


def quant_check(act, X, orc):
    xq_o, da_o = orc.quantize(X)
    N = X.shape[0]
    assert np.array_equal(host(act.xq), xq_o)
    assert np.array_equal(host(act.da)[:, :N].T, da_o)
    if act.xh is not None:
        assert np.array_equal(host(act.xh).astype(np.float32), xq_o.astype(np.float32))
    return xq_o, da_o


def chunk_sums(Po, raw, M, K):
    """Exact chunk sums from the oracle's sub-block partials Po [N][M][K/16]
    and the raw sub-block scales sc (int8 bytes 192..207 of each block)."""
    sc = raw.reshape(M, K // 256, 210)[:, :, 192:208].view(np.int8).reshape(M, K // 16)
    S = (Po.astype(np.int64) * sc.astype(np.int64)[None]).reshape(Po.shape[0], M, K // 32, 2)
    S = S.sum(-1)
    assert np.abs(S).max() < 2 ** 31
    return S.astype(np.int32)


SOURCES = ["raw", "wexp", "wh"]
TC_PATH = {"raw": "tc_raw", "wexp": "tc_wexp", "wh": "tc_wh"}


def expected_path(N, source, xq=True):
    """The path q6k_mmq takes: the few-token kernels for N <= 16, and on token
    groups of at most 32 given Xq, for N <= 32 whatever the source and for
    N <= 64 without resident planes; the tensor cores otherwise."""
    import q6_int8_mmq_gb300 as q6mod
    if N <= q6mod.SKINNY_MAX_N or (xq and (N <= q6mod.SKINNY_GROUP_N or (
            N <= q6mod.SKINNY_GROUPS_MAX_N and source != "wh"))):
        return "skinny"
    return TC_PATH[source]


def check_debug(D, Po, raw, M, K, tok=None, label=""):
    """Both debug outputs bit-exact: the sub-block partials against the
    oracle's P, the chunk sums against S formed from P and the raw scales
    (rows `tok` of the kernel's outputs when given)."""
    P, S = host(D.partials), host(D.chunk_sums)
    if tok is not None:
        P, S = P[tok], S[tok]
    assert np.array_equal(P, Po), f"{label}: sub-block partials differ"
    assert np.array_equal(S, chunk_sums(Po, raw, M, K)), f"{label}: chunk sums differ"


def run_gemm(q6, raw, X, M, K, source, partials=False):
    """Packs, quantises and runs the GEMM; with partials=True both debug
    outputs are requested."""
    w = q6.pack_weights(dev(raw), M, K, wexp=source == "wexp", wh=source == "wh")
    act = q6.quantize_act(dev(X))
    Y, path, D = q6.mmq(w, act, source=source, partials=partials, chunk_sums=partials)
    q6.sync_status()
    return w, act, Y, path, D


# --------------------------------------------------------------- failures ---

def test_bounded_wait_times_out_and_context_survives(q6):
    lib = q6.load()
    assert lib.q6_selftest_wait_timeout(50, None) == q6.Q6_OK
    with pytest.raises(q6.Q6Error) as ei:
        q6.sync_status()
    assert ei.value.code == q6.Q6_ETIMEOUT
    q6.sync_status()                    # the status word was cleared
    X = synth.activations(1, 4, 256)
    act = q6.quantize_act(dev(X))       # the context still works
    q6.sync_status()
    quant_check(act, X, oracle.get())


# -------------------------------------------------------------- quantiser ---

@pytest.mark.parametrize("N,K,frac", [(1, 256, 0.0), (8, 512, 0.0), (513, 4096, 0.0),
                                      (77, 11008, 0.01),
                                      # 16-element form with a partly idle last warp
                                      (1001, 1280, 0.02)])
def test_quantize_bitexact(q6, orc, N, K, frac):
    X = synth.activations(100 + N, N, K, outlier_frac=frac)
    X[0, 32:64] = 0.0                                   # all-zero block
    if N > 2:
        X[2, :32] = np.float32(1e-30)                   # tiny block
        X[1, :32] = 0.0
        X[1, 0] = 127.0
        X[1, 1:7] = [2.5, -2.5, 0.5, -0.5, 126.5, -126.5]   # exact halfway quotients
    act = q6.quantize_act(dev(X))
    q6.sync_status()
    quant_check(act, X, orc)


def hard_activations(seed, N, K, big=np.float32(1e36)):
    """Activations whose blocks put quotients on, one ulp beside and a little
    beside rounding ties (where the kernels leave the reciprocal for the exact
    division), have a subnormal scale (also taken exactly) or are scaled by
    `big`."""
    rng = np.random.default_rng(seed)
    X = synth.activations(seed + 493, N, K)
    blocks = X.reshape(N, K // 32, 32)
    kind = rng.integers(0, 4, size=blocks.shape[:2])
    for n, c in zip(*np.nonzero(kind == 1)):
        # amax 127 * s for a random power-of-two or odd scale s: the quotient
        # of x = (k + 1/2) * s and its float neighbours straddle the tie
        s = np.float32(rng.choice([1.0, 0.75, 3.0e-3, 17.0, 2.0 ** -20]))
        k = rng.integers(-126, 126, size=32).astype(np.float32)
        x = (k + np.float32(0.5)) * s
        step = rng.integers(-3, 4, size=32)
        x = np.array([np.nextafter(v, np.float32(np.inf) if d > 0 else np.float32(-np.inf))
                      if d else v for v, d in zip(x, step)], dtype=np.float32)
        x[0] = np.float32(127.0) * s
        blocks[n, c] = x
    for n, c in zip(*np.nonzero(kind == 2)):
        blocks[n, c] *= np.float32(1e-40)        # subnormal amax and scale
    for n, c in zip(*np.nonzero(kind == 3)):
        blocks[n, c] *= big                      # large values, normal scale
    return np.ascontiguousarray(blocks.reshape(N, K))


@pytest.mark.parametrize("N,K", [(3, 256), (300, 1024)])
def test_quantize_near_ties_and_tiny_scales(q6, orc, N, K):
    """Quotients on and beside rounding ties and subnormal block scales:
    bit-exact against the oracle."""
    X = hard_activations(7 + N, N, K)
    act = q6.quantize_act(dev(X))
    q6.sync_status()
    quant_check(act, X, orc)


def test_quantize_without_xq_and_gemm(q6, orc):
    """A prefill caller may skip the int8 Xq: Xh and da are the same, the
    tensor-core GEMM runs on them, and the few-token kernels refuse such
    activations (they read Xq)."""
    M, K, N = 256, 1024, 200
    raw = synth.q6k_raw_weights(0x51360C01, M, K)
    X = synth.activations(0x51360C02, N, K, outlier_frac=0.02)
    full = q6.quantize_act(dev(X))
    act = q6.quantize_act(dev(X), want_xq=False)
    q6.sync_status()
    assert act.xq is None
    assert np.array_equal(host(act.xh), host(full.xh))
    assert np.array_equal(host(act.da)[:, :N], host(full.da)[:, :N])
    w = q6.pack_weights(dev(raw), M, K)
    Y, path, _ = q6.mmq(w, act, source="raw")
    q6.sync_status()
    assert path == "tc_raw"
    xq_o, da_o = orc.quantize(X)
    check_y(host(Y), orc.mmq(raw, M, K, xq_o, da_o), "without Xq")
    few = q6.quantize_act(dev(X[:4]), want_xq=False)
    with pytest.raises(q6.Q6Error) as ei:
        q6.mmq(w, few, source="raw")
    assert ei.value.code == q6.Q6_EINVAL


def test_quantize_strided_input(q6, orc):
    import torch
    X = synth.activations(7, 33, 512)
    big = torch.zeros((33, 640), dtype=torch.float32, device="cuda")
    big[:, :512] = dev(X)
    act = q6.quantize_act(big[:, :512])
    q6.sync_status()
    quant_check(act, X, orc)


# ------------------------------------------------------------------- pack ---

@pytest.mark.parametrize("M,K", [(64, 256), (40, 512), (24, 768), (131, 1024)])
def test_pack_bitexact(q6, orc, M, K):
    raw = synth.q6k_raw_weights(200 + M, M, K)
    w = q6.pack_weights(dev(raw), M, K, wexp=True, wh=True)
    q6.sync_status()
    plane = host(w.plane)
    blocks = raw.reshape(M, K // 256, 210)
    r = lambda x: (x + 255) // 256 * 256
    ldm = (M + 3) // 4 * 4
    d_row = (K // 256 * 2 + 15) // 16 * 16
    qlh_sz, sc_sz, d_sz = M * K * 3 // 4, M * K // 16, M * d_row
    o_sc = r(qlh_sz)
    o_d = o_sc + r(sc_sz)
    o_dt = o_d + r(d_sz)
    assert plane.size == o_dt + r(K // 256 * ldm * 4)
    # the gaps that round each sub-plane up to 256 bytes are zero
    for a, b in ((qlh_sz, o_sc), (o_sc + sc_sz, o_d), (o_d + d_sz, o_dt),
                 (o_dt + K // 256 * ldm * 4, plane.size)):
        assert np.all(plane[a:b] == 0)
    # qlh: per half h of super-block b: ql[64h:64h+64] then qh[32h:32h+32]
    qlh = plane[:qlh_sz].reshape(M, K // 256, 2, 96)
    for h in range(2):
        assert np.array_equal(qlh[:, :, h, :64], blocks[:, :, 64 * h: 64 * h + 64])
        assert np.array_equal(qlh[:, :, h, 64:], blocks[:, :, 128 + 32 * h: 160 + 32 * h])
    sc = plane[o_sc:o_sc + sc_sz].view(np.int8).reshape(M, K // 256, 16)
    assert np.array_equal(sc, blocks[:, :, 192:208].view(np.int8))
    d_all = plane[o_d:o_d + d_sz].reshape(M, d_row)
    d = d_all[:, :K // 256 * 2].reshape(M, K // 256, 2)
    assert np.array_equal(d, blocks[:, :, 208:210])
    assert np.all(d_all[:, K // 256 * 2:] == 0)
    # d transposed to [K/256][ldm] as f32, rows M..ldm-1 zero
    dt = plane[o_dt:o_dt + K // 256 * ldm * 4].view(np.float32).reshape(K // 256, ldm)
    d_f64 = np.array([[orc.f16_to_f64(int(b[0]) | (int(b[1]) << 8)) for b in row] for row in d])
    assert np.array_equal(dt[:, :M].astype(np.float64), d_f64.T)
    assert np.all(dt[:, M:] == 0)
    v = orc.wexp(raw, M, K)
    assert np.array_equal(host(w.wexp), v)
    assert np.array_equal(host(w.wexp).astype(np.int64), restate.int_values(raw, M, K))
    # resident operand planes: W_hi = 16*floor(sc/16)*v, W_lo = (sc mod 16)*v
    sc16 = np.repeat(sc.reshape(M, K // 16).astype(np.int64), 16, axis=1)
    sh = np.floor_divide(sc16, 16)
    wh = host(w.wh).astype(np.float64)
    assert wh.shape == (2, M, K)
    assert np.array_equal(wh[0], 16 * sh * v)
    assert np.array_equal(wh[1], (sc16 - 16 * sh) * v)
    assert np.array_equal(wh[0] + wh[1], sc16 * v)
    # the unpack pass from the W_exp plane gives the same planes
    assert np.array_equal(host(q6.unpack_weights(w, from_wexp=True)).astype(np.float64), wh)
    assert np.array_equal(host(q6.unpack_weights(w)).astype(np.float64), wh)


def test_pack_from_host_memory(q6):
    """q6k_pack_weights reads the raw bytes from host memory (page-locked, or
    pageable where the device reads it) as well as from device memory: the
    same planes either way."""
    import torch
    M, K = 300, 1024
    raw = synth.q6k_raw_weights(0x51360D01, M, K)
    wd = q6.pack_weights(dev(raw), M, K, wexp=True, wh=True)
    for host_raw in (torch.from_numpy(raw).pin_memory(), torch.from_numpy(raw)):
        wh_ = q6.pack_weights(host_raw, M, K, wexp=True, wh=True)
        q6.sync_status()
        assert wh_.plane.is_cuda
        for a, b in ((wh_.plane, wd.plane), (wh_.wexp, wd.wexp), (wh_.wh, wd.wh)):
            assert torch.equal(a, b)
    # through the C ABI with a page-locked host pointer
    lib = q6.load()
    pinned = torch.from_numpy(raw).pin_memory()
    plane = torch.empty_like(wd.plane)
    rc = lib.q6k_pack_weights(ctypes.c_void_p(pinned.data_ptr()), M, K,
                              ctypes.c_void_p(plane.data_ptr()), None, None, None)
    assert rc == q6.Q6_OK, lib.q6_last_error().decode()
    torch.cuda.synchronize()
    assert torch.equal(plane, wd.plane)


# --------------------------------------------------------- GEMM, small ------

SMALL = [
    # (M, K, N) spanning tiles and ragged tails of both kernels
    (256, 512, 1), (256, 512, 4), (256, 512, 8), (200, 768, 16),      # skinny kernels
    (257, 512, 3), (129, 768, 16), (131, 2816, 2), (1000, 2560, 5),  # odd M, partial stages
    (3001, 768, 9),   # 20-row units: a partial second row group, a one-row last unit
    (48, 256, 6),     # one super-block per row, one row per unit
    (5000, 512, 16),  # more units than SMs: CTAs take two units each
    (128, 256, 17), (256, 512, 128), (200, 512, 129), (384, 768, 300),  # tensor-core kernel
    (130, 1024, 255), (64, 256, 40),
    (4800, 768, 5), (4800, 768, 12),  # 32-row units (the largest), 17-warp form
    (4800, 768, 24), (4800, 2304, 32),  # 32-row units, 17-32-token form; 9 super-blocks
    (1000, 1280, 20),  # 17-32-token form: 5 super-blocks, a last stage of one
]


@pytest.mark.parametrize("source", SOURCES)
@pytest.mark.parametrize("M,K,N", SMALL, ids=lambda v: str(v))
def test_mmq_small_bitexact_partials(q6, orc, M, K, N, source):
    raw = synth.q6k_raw_weights(300 + M + N, M, K)
    X = synth.activations(400 + M + N, N, K, outlier_frac=0.02)
    w, act, Y, path, D = run_gemm(q6, raw, X, M, K, source, partials=True)
    xq_o, da_o = quant_check(act, X, orc)
    Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
    assert path == expected_path(N, source)
    check_debug(D, Po, raw, M, K, label=f"{M}x{K}x{N} {source}")
    check_y(host(Y), Yo, f"{M}x{K}x{N}")
    # the fast (non-debug) variant gives the same Y
    Y2, _, _ = q6.mmq(w, act, source=source)
    q6.sync_status()
    check_y(host(Y2), Yo, "fast variant")


def _sweep_shapes(count=18, seed=0x5EED):
    """Seeded irregular shapes over the three kernel families: one or two
    tokens, 3..16 tokens, and the tensor-core GEMM (ragged M and N, 1..24
    super-blocks per row)."""
    rng = np.random.default_rng(seed)
    shapes = []
    for i in range(count):
        N = int([1, rng.integers(2, 17), rng.integers(17, 700)][i % 3])
        M = int(rng.integers(1, 3000))
        K = 256 * int(rng.integers(1, 25))
        shapes.append((M, K, N))
    return shapes


@pytest.mark.parametrize("M,K,N", _sweep_shapes(), ids=lambda v: str(v))
def test_mmq_seeded_shape_sweep(q6, orc, M, K, N):
    """Y within tolerance on every output of seeded irregular shapes (raw
    weight source), and bit-exact debug partials where they stay small."""
    raw = synth.q6k_raw_weights(900 + M + K + N, M, K)
    X = synth.activations(901 + M + K + N, N, K, outlier_frac=0.01)
    want_p = N * M * (K // 16) <= 20_000_000
    w, act, Y, path, D = run_gemm(q6, raw, X, M, K, "raw", partials=want_p)
    xq_o, da_o = quant_check(act, X, orc)
    if want_p:
        Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
        check_debug(D, Po, raw, M, K, label=f"{M}x{K}x{N}")
    else:
        Yo = orc.mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"{M}x{K}x{N}")
    Y2, _, _ = q6.mmq(w, act, source="raw")
    q6.sync_status()
    check_y(host(Y2), Yo, f"{M}x{K}x{N} fast")


@pytest.mark.parametrize("M,K,N", [(1016, 768, 2555), (4096, 2048, 16), (3001, 768, 9),
                                    (2059, 1024, 1), (4096, 2048, 40)], ids=lambda v: str(v))
def test_mmq_deterministic(q6, M, K, N):
    """Repeated calls give bit-identical Y: the split last round of the
    tensor-core GEMM adds two halves onto zero, the K parts of a call with few
    tiles are added in a fixed order, and the few-token kernels reduce in a
    fixed order."""
    import torch
    raw = synth.q6k_raw_weights(1200 + M + N, M, K)
    X = synth.activations(1201 + M + N, N, K, outlier_frac=0.01)
    w = q6.pack_weights(dev(raw), M, K, wh=True)
    act = q6.quantize_act(dev(X))
    Y0, _, _ = q6.mmq(w, act, source="wh")
    for _ in range(3):
        Y1, _, _ = q6.mmq(w, act, source="wh")
        q6.sync_status()
        assert torch.equal(Y0, Y1)


@pytest.mark.parametrize("source", ["raw", "wh"])
@pytest.mark.parametrize("M,K,N,splits", [(4096, 11008, 17, 4), (4096, 11008, 100, 4),
                                          (4096, 2048, 200, 2), (1000, 768, 40, 3),
                                          (300, 512, 130, 2)], ids=lambda v: str(v))
def test_mmq_splitk_few_tiles(q6, orc, M, K, N, splits, source):
    """Few tiles (at most half the SMs): each tile is split into K parts whose
    partial sums a second kernel adds in order. Y within tolerance of the
    oracle on every output, the debug partials bit-exact, the planned split
    as expected, and the same Y (up to rounding) as without the split (a
    workspace without room for the partial sums)."""
    import torch
    assert q6.tc_part_bytes(M, K, N) == splits * N * M * 4
    raw = synth.q6k_raw_weights(1300 + M + N, M, K)
    X = synth.activations(1301 + M + N, N, K, outlier_frac=0.01)
    w = q6.pack_weights(dev(raw), M, K, wh=source == "wh")
    act = q6.quantize_act(dev(X), want_xq=False)   # no Xq: the tensor cores at any N > 16
    xq_o, da_o = orc.quantize(X)
    assert np.array_equal(host(act.da)[:, :N].T, da_o)
    want_p = N * M * (K // 16) <= 40_000_000
    Y, path, D = q6.mmq(w, act, source=source, partials=want_p, chunk_sums=want_p)
    q6.sync_status()
    assert path == TC_PATH[source]
    if want_p:
        Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
        check_debug(D, Po, raw, M, K, label=f"splitk {M}x{K}x{N}")
    else:
        Yo = orc.mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"splitk {M}x{K}x{N} {source}")
    # unsplit: a workspace with room for the unpacked planes only
    ws = torch.empty(4 * M * K if source == "raw" else 256, dtype=torch.uint8, device="cuda")
    Y1, _, _ = q6.mmq(w, act, source=source, workspace=ws)
    q6.sync_status()
    check_y(host(Y1), Yo, f"unsplit {M}x{K}x{N} {source}")
    assert torch.allclose(Y, Y1, rtol=1e-5, atol=1e-5 * float(Y1.abs().max()))


@pytest.mark.parametrize("source", ["raw", "wexp", "wh"])
@pytest.mark.parametrize("M,K,N", [(4096, 11008, 17), (1000, 2816, 20), (300, 768, 32),
                                   (300, 768, 33), (700, 1280, 50), (300, 768, 64),
                                   (300, 768, 65), (4096, 11008, 32), (1000, 2816, 46),
                                   (300, 768, 96), (300, 768, 97)],
                         ids=lambda v: str(v))
def test_mmq_token_groups(q6, orc, M, K, N, source):
    """Given Xq, 17..32 tokens run the few-token kernels whatever the source
    and 33..96 tokens without resident planes, on token groups of at most 32
    (the 17..32-token form of the MMA kernel; offset rows of Xq, Y and the
    debug outputs, offset columns of da; a last group of one or two tokens
    on the dp4a kernel): bit-exact partials and Y within tolerance; 97
    tokens, and 33 and more on resident planes, take the tensor cores. The
    same Y, up to rounding, as the tensor cores on the same activations
    without Xq."""
    import torch
    raw = synth.q6k_raw_weights(1400 + M + N, M, K)
    X = synth.activations(1401 + M + N, N, K, outlier_frac=0.01)
    w = q6.pack_weights(dev(raw), M, K, wexp=source == "wexp", wh=source == "wh")
    act = q6.quantize_act(dev(X))
    xq_o, da_o = quant_check(act, X, orc)
    want_p = N * M * (K // 16) <= 40_000_000
    Y, path, D = q6.mmq(w, act, source=source, partials=want_p, chunk_sums=want_p)
    q6.sync_status()
    assert path == expected_path(N, source)
    if want_p:
        Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
        check_debug(D, Po, raw, M, K, label=f"groups {M}x{K}x{N}")
    else:
        Yo = orc.mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"groups {M}x{K}x{N} {source}")
    act_tc = q6.quantize_act(dev(X), want_xq=False)
    Yt, tpath, _ = q6.mmq(w, act_tc, source=source)
    q6.sync_status()
    assert tpath == TC_PATH[source]
    assert torch.allclose(Y, Yt, rtol=1e-5, atol=1e-5 * float(Yt.abs().max()))


def test_mmq_degenerate_inputs(q6, orc):
    M, K, N = 128, 512, 130
    blk = np.zeros(210, np.uint8)
    blk[128:192] = 0xAA                     # every code 32: all values zero
    blk[192:208] = 7
    blk[208:210] = [0x00, 0x3C]
    raw = np.tile(blk, (M, K // 256))
    X = synth.activations(5, N, K)
    for n in (N, 3):                         # tensor-core and skinny kernels
        _, _, Y, _, _ = run_gemm(q6, raw, X[:n], M, K, "raw")
        assert np.all(host(Y) == 0.0)
    raw = synth.q6k_raw_weights(6, M, K).reshape(-1, 210).copy()
    raw[:, 208:210] = 0                      # d = 0 everywhere
    _, _, Y, _, _ = run_gemm(q6, raw.reshape(M, -1), X, M, K, "wexp")
    assert np.all(host(Y) == 0.0)
    X0 = X.copy()
    X0[5] = 0.0                              # a zero token
    raw = synth.q6k_raw_weights(7, M, K)
    _, _, Y, _, _ = run_gemm(q6, raw, X0, M, K, "wh")
    assert np.all(host(Y)[5] == 0.0)


@pytest.mark.parametrize("N", [128, 4])
def test_mmq_extreme_chunk_sums_exact(q6, orc, N):
    """Chunk sums at the edge of the exact range: |v| = 32, |xq| = 127 and the
    sub-block scales whose W_hi part is largest (sc = -128, -113: 16*floor(sc/16)
    = -128), alone and mixed with positive scales and signs, so the MMA
    accumulator passes through partial sums close to 2^24."""
    M, K = 128, 512
    nblk = M * (K // 256)
    blocks = np.zeros((nblk, 210), np.uint8)
    rng = np.random.default_rng(11)
    codes_max = rng.random(nblk) < 0.5
    codes_max[0] = False                                            # block 0: every v = -32
    blocks[:, 0:192] = np.where(codes_max[:, None], 0xFF, 0x00)   # every code 63 or 0
    scs = np.array([-128, -113, 127, -1, -128, -128, 112, -113], np.int8)
    for i in range(nblk):
        blocks[i, 192:208] = scs[(i + np.arange(16)) % len(scs)].view(np.uint8)
    blocks[:, 208:210] = [0x00, 0x3C]                               # d = 1.0
    raw = blocks.reshape(M, -1)
    X = np.ones((N, K), np.float32)
    X[1::2] *= -1.0                                                 # +-1 rows: xq = +-127
    X[0, 256:] = np.where(np.arange(256) % 3 == 0, -1.0, 1.0)
    for source in ("raw", "wh"):
        w, act, Y, path, D = run_gemm(q6, raw, X, M, K, source, partials=True)
        xq_o, da_o = quant_check(act, X, orc)
        assert np.abs(xq_o).min() == 127
        Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
        S = chunk_sums(Po, raw, M, K)
        assert np.abs(S).max() == 32 * 128 * 32 * 127                # the bound is reached
        check_debug(D, Po, raw, M, K, label=f"extreme {source}")
        check_y(host(Y), Yo, f"extreme N={N}")


@pytest.mark.parametrize("source", ["raw", "wh"])
def test_mmq_split_last_round(q6, orc, source):
    """160 tiles of 128 x 128 on 152 SMs: the last 8 tiles (the last weight
    band, token tiles 12-19) are each computed as two halves of their
    super-blocks (1 and 2 of K/256 = 3) on two SMs and added into Y after a
    zeroing kernel. The split tiles hold the ragged last token tile and the
    ragged last band (M = 1016: a 56-column half that takes the scalar adds).
    Y starts as NaN; sampled tokens inside and outside the split tiles are
    checked against the oracle over all columns, with bit-exact partials."""
    import torch
    M, K, N = 1016, 768, 2555
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = ((N + 127) // 128) * ((M + 127) // 128)
    rem = tiles % sms
    split = tiles > sms and rem > 0 and 2 * rem <= sms
    assert q6.mmq_launches(M, K, N, True) == 1 + int(split)
    assert q6.mmq_launches(M, K, N, False) == 2 + int(split)
    if sms == 152:
        assert split
    raw = synth.q6k_raw_weights(0x51360A01, M, K)
    X = synth.activations(0x51360A02, N, K, outlier_frac=0.02)
    w = q6.pack_weights(dev(raw), M, K, wh=source == "wh")
    act = q6.quantize_act(dev(X))
    xq_o, da_o = quant_check(act, X, orc)
    tok = sampled_tokens(N, extra=(1535, 1536, 1700, 2047, 2300, 2431, 2432, 2500))
    for partials in (False, True):
        Y = torch.full((N, M), float("nan"), dtype=torch.float32, device="cuda")
        Y, path, D = q6.mmq(w, act, Y=Y, source=source, partials=partials, chunk_sums=partials)
        q6.sync_status()
        assert path == TC_PATH[source]
        Yh = host(Y)
        assert np.all(np.isfinite(Yh)), "a split tile was not zeroed or not written"
        if partials:
            Yo, Po = orc.mmq(raw, M, K, xq_o[tok], da_o[tok], partials=True)
            check_debug(D, Po, raw, M, K, tok=tok, label=f"split {source}")
        else:
            Yo = orc.mmq(raw, M, K, xq_o[tok], da_o[tok])
        check_y(Yh[tok], Yo, f"split {source} partials={partials}")


def test_mmq_empty(q6):
    import torch
    M, K = 128, 256
    raw = synth.q6k_raw_weights(8, M, K)
    w = q6.pack_weights(dev(raw), M, K)
    act = q6.alloc_activations(0, K)
    Y, path, _ = q6.mmq(w, act, Y=torch.empty((0, M), device="cuda"))
    q6.sync_status()
    assert path == "none"


@pytest.mark.parametrize("M,K,N,kind", [
    (328, 1024, 1, "raw"), (328, 1024, 2, "raw"), (328, 1024, 7, "raw"),  # skinny kernels
    (328, 1024, 20, "raw"),                               # few-token kernels, two token groups
    (1016, 768, 2555, "raw"), (1016, 768, 2555, "wh"),   # tensor-core GEMM, split last round
    (256, 512, 40, "mma_sync")], ids=lambda v: str(v))
def test_mmq_strided_unaligned_output(q6, orc, M, K, N, kind):
    """Y as a view with an odd row stride (M + 37 floats) starting 4 bytes past
    a 16-byte boundary: every kernel family takes its scalar stores, writes
    Y[:N, :M] and leaves every other float of the buffer untouched."""
    import torch
    raw = synth.q6k_raw_weights(0x51360B01 + N, M, K)
    X = synth.activations(0x51360B02 + N, N, K, outlier_frac=0.01)
    w = q6.pack_weights(dev(raw), M, K, wh=kind == "wh", wexp=kind == "mma_sync")
    act = q6.quantize_act(dev(X))
    xq_o, da_o = quant_check(act, X, orc)
    ldy = M + 37
    buf = torch.full((N * ldy + 1,), float("nan"), dtype=torch.float32, device="cuda")
    Y = buf[1:].view(N, ldy)[:, :M]
    assert Y.data_ptr() % 16 == 4 and Y.stride(0) == ldy
    if kind == "mma_sync":
        Y2, path, _ = q6.mmq_mma_sync(w, act, Y=Y)
    else:
        Y2, path, _ = q6.mmq(w, act, Y=Y, source=kind)
        assert path == expected_path(N, kind)
    q6.sync_status()
    assert Y2.data_ptr() == Y.data_ptr()
    b = host(buf)
    assert np.isnan(b[0]) and np.all(np.isnan(b[1:].reshape(N, ldy)[:, M:]))
    Yh = host(Y)
    assert np.all(np.isfinite(Yh))
    tok = sampled_tokens(N, extra=(1535, 1536, 2047, 2432, 2500))
    check_y(Yh[tok], orc.mmq(raw, M, K, xq_o[tok], da_o[tok]), f"strided {M}x{K}x{N} {kind}")


def test_mmq_refuses_mismatched_buffers(q6):
    """An output or activation buffer the kernels would misread is refused by
    the binding before anything is launched, and the path still works after."""
    import torch
    M, K, N = 256, 512, 5
    raw = synth.q6k_raw_weights(0x51360B10, M, K)
    w = q6.pack_weights(dev(raw), M, K)
    X = dev(synth.activations(0x51360B11, N, K))
    act = q6.quantize_act(X)
    for Y in (torch.empty((N, M - 1), device="cuda"),                # too narrow
              torch.empty((M, N), device="cuda").t(),                # columns not contiguous
              torch.empty((N, M), dtype=torch.float16, device="cuda"),
              torch.empty((N, M))):                                  # host memory
        with pytest.raises(q6.Q6Error):
            q6.mmq(w, act, Y=Y)
    with pytest.raises(q6.Q6Error):
        q6.quantize_act(X, out=q6.alloc_activations(N + 1, K))
    with pytest.raises(q6.Q6Error):
        q6.mmq(w, q6.quantize_act(X[:, :256].contiguous()))         # K does not match
    with pytest.raises(dataclasses.FrozenInstanceError):
        act.xq = torch.empty((N + 1, K), dtype=torch.int8, device="cuda")
    Y, path, _ = q6.mmq(w, act)
    q6.sync_status()
    assert path == "skinny" and bool(torch.isfinite(Y).all())


@pytest.mark.parametrize("M,K,N", [(4096, 11008, 1), (4096, 11008, 2), (4096, 4096, 2),
                                   (1, 256, 1), (131, 2816, 2), (5003, 768, 2), (2059, 1024, 1)],
                         ids=lambda v: str(v))
def test_mmq_f32_equals_quantise_then_mmq(q6, orc, M, K, N):
    """The fused one/two-token call gives bit for bit the Y of quantize_act
    followed by mmq (the same codes, dot products and order), on ordinary
    activations and on blocks at and beside rounding ties, with subnormal and
    very large scales; Y within tolerance of the oracle on every output. The
    shapes cover the full-size weights, one row, more rows than warps and
    one super-block per row."""
    import torch
    raw = synth.q6k_raw_weights(0x51360C01 + M + N, M, K)
    w = q6.pack_weights(dev(raw), M, K)
    X0 = synth.activations(0x51360C02 + K + N, N, K, outlier_frac=0.01)
    for X in (X0, hard_activations(0x51360C03 + N, N, K, big=np.float32(1e30))):
        Xd = dev(X)
        Y, path = q6.mmq_f32(w, Xd)
        act = q6.quantize_act(Xd)
        Y2, path2, _ = q6.mmq(w, act)
        q6.sync_status()
        assert path == "skinny_fused" and path2 == "skinny"
        assert torch.equal(Y, Y2), "fused and separate quantisation disagree"
    act = q6.quantize_act(dev(X0))
    xq_o, da_o = quant_check(act, X0, orc)
    Yo = orc.mmq_all(raw, M, K, xq_o, da_o) if M * K > 1 << 22 else orc.mmq(raw, M, K, xq_o, da_o)
    Y, _ = q6.mmq_f32(w, dev(X0))
    q6.sync_status()
    check_y(host(Y), Yo, f"fused {M}x{K}x{N}")


@pytest.mark.parametrize("N", [1, 9, 130])
def test_mmq_long_rows(q6, orc, N):
    """Rows of K = 65,536 (256 super-blocks, several times the longest
    workload) through the dp4a, few-token and tensor-core kernels: Y within
    tolerance of the oracle on every output."""
    M, K = 128, 65536
    raw = synth.q6k_raw_weights(0x51360C31 + N, M, K)
    X = synth.activations(0x51360C32 + N, N, K, outlier_frac=0.01)
    w, act, Y, path, _ = run_gemm(q6, raw, X, M, K, "raw")
    assert path == ("skinny" if N <= q6.SKINNY_MAX_N else "tc_raw")
    xq_o, da_o = quant_check(act, X, orc)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), f"long rows N={N}")


@pytest.mark.parametrize("M,K,N", [(20000, 512, 1), (20000, 512, 5), (20000, 512, 200),
                                   (128, 256, 20000)], ids=lambda v: str(v))
def test_mmq_large_extents(q6, orc, M, K, N):
    """Many weight rows (20,000: several rounds of tiles, a ragged last band,
    more rows than the few-token kernels' warps and units) and many tokens
    (20,000 against one band): Y within tolerance of the oracle on every
    output."""
    raw = synth.q6k_raw_weights(0x51360C41 + M + N, M, K)
    X = synth.activations(0x51360C42 + M + N, N, K, outlier_frac=0.01)
    w, act, Y, path, _ = run_gemm(q6, raw, X, M, K, "raw")
    assert path == ("skinny" if N <= q6.SKINNY_MAX_N else "tc_raw")
    xq_o, da_o = quant_check(act, X, orc)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), f"large {M}x{K}x{N}")


@pytest.mark.parametrize("K,N", [(103168, 2), (206592, 1)], ids=lambda v: str(v))
def test_mmq_f32_largest_k(q6, orc, K, N):
    """The largest K whose codes and scales fit the fused kernel's shared
    memory for N tokens (232,128 and 232,416 of 232,448 bytes): the same Y as
    the separate calls, within tolerance of the oracle; one more super-block
    is refused."""
    import torch
    M = 96
    raw = synth.q6k_raw_weights(0x51360C21 + N, M, K)
    X = synth.activations(0x51360C22 + N, N, K, outlier_frac=0.01)
    w = q6.pack_weights(dev(raw), M, K)
    Xd = dev(X)
    Y, path = q6.mmq_f32(w, Xd)
    act = q6.quantize_act(Xd)
    Y2, _, _ = q6.mmq(w, act)
    q6.sync_status()
    assert path == "skinny_fused" and torch.equal(Y, Y2)
    xq_o, da_o = quant_check(act, X, orc)
    check_y(host(Y), orc.mmq(raw, M, K, xq_o, da_o), f"fused K={K} N={N}")
    K2 = K + 256
    w2 = q6.pack_weights(dev(synth.q6k_raw_weights(0x51360C23, M, K2)), M, K2)
    with pytest.raises(q6.Q6Error):
        q6.mmq_f32(w2, dev(synth.activations(0x51360C24, N, K2)))


def test_mmq_f32_strided_input_and_output(q6):
    """X with a wider row stride, Y with an odd row stride at an unaligned
    address: the floats between Y's rows stay untouched, the result equals
    the separate path's."""
    import torch
    M, K, N = 328, 1024, 2
    raw = synth.q6k_raw_weights(0x51360C11, M, K)
    w = q6.pack_weights(dev(raw), M, K)
    big = torch.full((N, K + 64), float("nan"), dtype=torch.float32, device="cuda")
    big[:, :K] = dev(synth.activations(0x51360C12, N, K))
    Xv = big[:, :K]
    ldy = M + 37
    buf = torch.full((N * ldy + 1,), float("nan"), dtype=torch.float32, device="cuda")
    Yv = buf[1:].view(N, ldy)[:, :M]
    Y, path = q6.mmq_f32(w, Xv, Y=Yv)
    Y2, _, _ = q6.mmq(w, q6.quantize_act(Xv))
    q6.sync_status()
    assert path == "skinny_fused" and Y.data_ptr() == Yv.data_ptr()
    assert torch.equal(Yv, Y2)
    b = host(buf)
    assert np.isnan(b[0]) and np.all(np.isnan(b[1:].reshape(N, ldy)[:, M:]))
    with pytest.raises(q6.Q6Error):
        q6.mmq_f32(w, dev(synth.activations(0x51360C13, 3, K)))   # three tokens


# ------------------------------------------------------ full-size workloads --

def sampled_tokens(N, extra=()):
    idx = {0, 1, N - 1, N // 2, (N // 128) * 128, max(0, (N // 128) * 128 - 1), *extra}
    return np.array(sorted(i for i in idx if 0 <= i < N))


def check_full(q6, orc, raw, X, M, K, source, label):
    """Every output of a full-size GEMM against the oracle (run over disjoint
    weight-row ranges on the host cores)."""
    w, act, Y, path, P = run_gemm(q6, raw, X, M, K, source)
    xq_o, da_o = quant_check(act, X, orc)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), label)
    return w, act, path


@pytest.mark.parametrize("source", SOURCES)
def test_attn_v_full(q6, orc, source):
    raw, X, cfg = synth.workload("attn_v")
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    w, act, path = check_full(q6, orc, raw, X, M, K, source, "attn_v")
    assert path == TC_PATH[source]
    # debug partials of four tokens, bit-exact
    Y, _, D = q6.mmq(w, act, source=source, partials=True, chunk_sums=True)
    q6.sync_status()
    tok = np.array([0, 129, 300, N - 1])
    xq_o, da_o = orc.quantize(X[tok])
    _, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
    check_debug(D, Po, raw, M, K, tok=tok, label=f"attn_v {source}")


@pytest.mark.parametrize("source", SOURCES)
def test_ffn_down_full(q6, orc, source):
    raw, X, cfg = synth.workload("ffn_down")
    check_full(q6, orc, raw, X, cfg["M"], cfg["K"], source, "ffn_down")


def test_ffn_down_debug_partials_sampled_tokens(q6, orc):
    """The full ffn_down weights (4096 x 11008) against 136 sampled tokens of
    its activation stream (tile edges, the ragged last tile, outlier-heavy
    rows): enough tokens for the tensor-core path, whose sub-block partials
    P [136][4096][688] and chunk sums are compared bit-exactly with the
    oracle; each token is quantised on its own, so the sample is the same
    computation as in the full GEMM. Y within tolerance on every output."""
    raw, X, cfg = synth.workload("ffn_down")
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    tok = np.unique(np.concatenate([sampled_tokens(N, extra=(127, 128, 255, 256, 3199, 3200)),
                                    np.linspace(0, N - 1, 136, dtype=np.int64)]))[:136]
    assert tok.size > q6.SKINNY_MAX_N
    Xs = np.ascontiguousarray(X[tok])
    for source in ("raw", "wh"):
        w, act, Y, path, D = run_gemm(q6, raw, Xs, M, K, source, partials=True)
        assert path == TC_PATH[source]
        xq_o, da_o = quant_check(act, Xs, orc)
        Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
        check_debug(D, Po, raw, M, K, label=f"ffn_down sampled tokens {source}")
        check_y(host(Y), Yo, f"ffn_down sampled tokens {source}")


@pytest.mark.parametrize("M,K,N", [(256, 512, 8), (200, 768, 129), (384, 768, 300), (130, 1024, 1)],
                         ids=lambda v: str(v))
def test_mma_sync_comparison_path(q6, orc, M, K, N):
    """The legacy mma.sync path: bit-exact debug partials and Y within tolerance."""
    raw = synth.q6k_raw_weights(500 + M + N, M, K)
    X = synth.activations(600 + M + N, N, K, outlier_frac=0.02)
    w = q6.pack_weights(dev(raw), M, K, wexp=True)
    act = q6.quantize_act(dev(X))
    Y, path, D = q6.mmq_mma_sync(w, act, partials=True, chunk_sums=True)
    q6.sync_status()
    assert path == "sync_wexp"
    xq_o, da_o = quant_check(act, X, orc)
    Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
    check_debug(D, Po, raw, M, K, label=f"mma.sync {M}x{K}x{N}")
    check_y(host(Y), Yo, f"mma.sync {M}x{K}x{N}")
    Y2, _, _ = q6.mmq_mma_sync(w, act)
    q6.sync_status()
    check_y(host(Y2), Yo, "mma.sync fast variant")


def test_mma_sync_ffn_down_full(q6, orc):
    raw, X, cfg = synth.workload("ffn_down")
    M, K = cfg["M"], cfg["K"]
    w = q6.pack_weights(dev(raw), M, K, wexp=True)
    act = q6.quantize_act(dev(X))
    Y, path, _ = q6.mmq_mma_sync(w, act)
    q6.sync_status()
    xq_o, da_o = quant_check(act, X, orc)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), "mma.sync ffn_down")


@pytest.mark.parametrize("name", ["pages_ffn_down", "pages_attn_v"])
def test_pages_shapes_full(q6, orc, name):
    """The shapes the pages measure (3584 x 18944 and 512 x 3584, N = 3325)."""
    raw, X, cfg = synth.workload(name)
    w, act, path = check_full(q6, orc, raw, X, cfg["M"], cfg["K"], "raw", name)
    assert path == "tc_raw"


@pytest.mark.parametrize("weight", ["ffn_down", "attn_v"])
@pytest.mark.parametrize("N", synth.SKINNY_N)
def test_skinny_full(q6, orc, weight, N):
    raw, X, cfg = synth.skinny_workload(weight, N)
    M, K = cfg["M"], cfg["K"]
    w, act, Y, path, D = run_gemm(q6, raw, X, M, K, "raw", partials=True)
    assert path == "skinny"
    xq_o, da_o = quant_check(act, X, orc)
    Yo, Po = orc.mmq(raw, M, K, xq_o, da_o, partials=True)
    check_debug(D, Po, raw, M, K, label=f"skinny {weight} N={N}")
    check_y(host(Y), Yo, f"skinny {weight} N={N}")
    Y2, _, _ = q6.mmq(w, act, source="raw")            # the fast kernel of this N
    q6.sync_status()
    check_y(host(Y2), Yo, f"skinny {weight} N={N} fast")


@pytest.mark.parametrize("layer", [0, 31])
def test_sweep_layers(q6, orc, layer):
    raw_v, raw_d = synth.sweep_layer(layer)
    X_v, X_d = synth.sweep_activations()
    check_full(q6, orc, raw_v, X_v, 4096, 4096, "raw", f"sweep layer {layer} attn_v")
    check_full(q6, orc, raw_d, X_d, 4096, 11008, "raw", f"sweep layer {layer} ffn_down")


@pytest.mark.parametrize("fmt", ["q6_K", "q4_K"])
def test_few_token_gemm_sees_the_previous_kernels_writes(q6, orc, fmt):
    """The few-token GEMMs start as programmatic dependent launches and wait
    for the previous kernel in the stream before they touch global memory.
    Here each GEMM follows, with no synchronisation, a kernel that rewrote
    its inputs: two weight matrices packed in turn into the same plane
    buffer, and two activation rows quantised in turn into the same buffers
    (the quantiser lets its dependants start early). Every Y must belong to
    the weights and activations of its own turn: 1, 5 and 16 tokens (dp4a,
    f16 with one and two token tiles), and 24 (token groups)."""
    import torch
    q4 = fmt == "q4_K"
    M, K = 1000, 2048
    lib = q6.load()
    if q4:
        raws = [synth.q4k_raw_weights(0x51360C01 + i, M, K) for i in range(2)]
        W = q6.q4k_pack_weights(dev(raws[0]), M, K)
    else:
        raws = [synth.q6k_raw_weights(0x51360C01 + i, M, K) for i in range(2)]
        W = q6.pack_weights(dev(raws[0]), M, K)
    raw_d = [dev(r) for r in raws]
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for N in (1, 5, 16, 24):
        Xs = [synth.activations(0x51360C10 + 4 * N + i, N, K) for i in range(2)]
        Xd = [dev(x) for x in Xs]
        act = q6.alloc_activations(N, K, torch.device("cuda"), want_xh=False, want_us=q4)
        expect = {}
        for i in range(2):
            xq_o, da_o = orc.quantize(Xs[i])
            for j in range(2):
                expect[i, j] = (orc.q4k_mmq(raws[j], M, K, xq_o, da_o) if q4
                                else orc.mmq(raws[j], M, K, xq_o, da_o))
        torch.cuda.synchronize()
        got = []
        for it in range(8):
            i, j = it % 2, (it // 2) % 2   # activations of turn i, weights of turn j
            rc = (lib.q4k_pack_weights(q6._ptr(raw_d[j]), M, K, q6._ptr(W.plane), None, s) if q4
                  else lib.q6k_pack_weights(q6._ptr(raw_d[j]), M, K, q6._ptr(W.plane), None,
                                            None, s))
            assert rc == 0
            q6.quantize_act(Xd[i], out=act)
            Y, path, _ = (q6.q4k_mmq(W, act) if q4 else q6.mmq(W, act, source="raw"))
            assert path == ("q4k_skinny" if q4 else "skinny")
            got.append(((i, j), Y.clone()))
        q6.sync_status()
        for key, Y in got:
            check_y(host(Y), expect[key], f"{fmt} N={N} turn {key}")


@pytest.mark.parametrize("M,K", [(4096, 11008), (131, 2816), (64, 103168), (64, 103424)],
                         ids=lambda v: str(v))
def test_two_tokens_staged_equals_plain(q6, orc, M, K):
    """Two tokens without debug outputs run the kernel that stages the codes
    and scales in shared memory (up to K = 103,168, the largest its shared
    memory holds; one super-block beyond, the plain dp4a kernel): Y bit for
    bit that of the plain kernel (the debug run), within tolerance of the
    oracle; also as the last group of 34 tokens."""
    import torch
    raw = synth.q6k_raw_weights(0x51362401 + M + K, M, K)
    w = q6.pack_weights(dev(raw), M, K)
    for N in (2, 34):
        X = synth.activations(0x51362402 + K + N, N, K, outlier_frac=0.01)
        act = q6.quantize_act(dev(X))
        Y, path, D = q6.mmq(w, act, partials=True)
        Y2, path2, _ = q6.mmq(w, act)
        q6.sync_status()
        assert path == path2 == "skinny"
        assert torch.equal(Y, Y2)
        xq_o, da_o = quant_check(act, X, orc)
        Yo = orc.mmq_all(raw, M, K, xq_o, da_o) if M * K > 1 << 22 else orc.mmq(raw, M, K,
                                                                               xq_o, da_o)
        check_y(host(Y2), Yo, f"two tokens staged {M}x{K}x{N}")
