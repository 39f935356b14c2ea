"""Parity of the q4_K GEMM with the CPU oracle (needs a GB300).

The q4_K line of the pages ("r18: Load-time B pre-expansion", Sec. 1 and 3.2;
the two-term rescale of "r38 -- q6_K BT-style raw-byte mma kernel", Sec.
2.2). Integer results (the packed plane, the activation block sums, the debug
partials P = sum over a 32-element sub-block of q * xq) must be bit-exact; Y
must satisfy max|Y - Yo| <= 1e-3 * max|Yo| and sum|Y - Yo| / sum|Yo| <= 1e-5,
as for q6_K.
"""
import numpy as np
import pytest

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
    assert err.max() / scale <= MAX_REL, f"{label}: max error {err.max() / scale:.3e}"
    assert err.sum() / np.abs(Yo).sum() <= NORMWISE, f"{label}: normwise error"


def tf32_pairs(v):
    """[rows, K/32] f32 -> [rows, ldus]: per super-block the hi parts of its 8
    values (low 13 mantissa bits cleared), then the lo parts v - hi; an odd
    super-block count padded with 16 zeros (the GEMM's min-term operand)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    hi = (v.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    lo = v - hi
    rows, nc = v.shape
    nsb = nc // 8
    out = np.zeros((rows, 32 * ((nsb + 1) // 2)), dtype=np.float32)
    pairs = np.concatenate([hi.reshape(rows, nsb, 8), lo.reshape(rows, nsb, 8)], axis=2)
    out[:, :16 * nsb] = pairs.reshape(rows, 16 * nsb)
    return out


def test_tf32_pairs_are_exact_splits():
    """hi + lo == v; hi keeps 11 significant bits; a value with at most 17
    significant bits (dmin * m) leaves a lo of at most 6."""
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((3, 24)) * 10.0 ** rng.integers(-6, 6, (3, 24))).astype(np.float32)
    p = tf32_pairs(v)
    hi, lo = p[:, :32].reshape(3, 2, 16)[:, :, :8], p[:, :32].reshape(3, 2, 16)[:, :, 8:]
    assert np.array_equal(hi.reshape(3, 16) + lo.reshape(3, 16), v[:, :16])
    assert np.all((hi.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    assert p.shape == (3, 64) and np.all(p[:, 48:] == 0)
    dmin = np.float32(np.float16(0.00213))
    mv = np.float32(dmin * np.float32(61))
    q = tf32_pairs(np.full((1, 8), mv, dtype=np.float32))
    lo1 = q[0, 8]
    m, e = np.frexp(np.float64(lo1))
    assert lo1 != 0 and (m * 2 ** 6) == np.round(m * 2 ** 6)


def quantize(q6, orc, X):
    """GPU activations with block sums, checked bit-exactly against the oracle's
    codes and scales; us against the pairs of da * S rounded to f32 once."""
    act = q6.quantize_act(dev(X), want_us=True)
    q6.sync_status()
    xq_o, da_o = orc.quantize(X)
    N = X.shape[0]
    assert np.array_equal(host(act.xq), xq_o)
    assert np.array_equal(host(act.da)[:, :N].T, da_o)
    S = xq_o.astype(np.int64).reshape(N, -1, 32).sum(-1).astype(np.float32)
    assert np.array_equal(host(act.us), tf32_pairs(da_o * S))
    return act, xq_o, da_o


@pytest.mark.parametrize("N,K", [(3, 256), (700, 1024), (77, 11008), (5, 768)])
def test_quantize_block_sums(q6, orc, N, K):
    X = synth.activations(0x51361001 + N, N, K, outlier_frac=0.01)
    X[0, 32:64] = 0.0
    quantize(q6, orc, X)


@pytest.mark.parametrize("M,K", [(64, 256), (131, 768), (300, 1024), (40, 1280)])
def test_q4k_pack_bitexact(q6, orc, M, K):
    raw = synth.q4k_raw_weights(0x51361101 + M, M, K)
    w = q6.q4k_pack_weights(dev(raw), M, K, wq=True)
    q6.sync_status()
    plane = host(w.plane)
    r = lambda x: (x + 255) // 256 * 256
    ldm = (M + 3) // 4 * 4
    nsb, nc = K // 256, K // 32
    o_sc = r(M * K // 2)
    o_mn = o_sc + r(M * nc)
    o_dt = o_mn + r(M * nc)
    o_mv = o_dt + r(nsb * ldm * 4)
    ldus = 32 * ((nsb + 1) // 2)
    o_dd = o_mv + r(M * ldus * 4)
    assert plane.size == o_dd + r(M * nsb * 8)
    for a, b in ((M * K // 2, o_sc), (o_sc + M * nc, o_mn), (o_mn + M * nc, o_dt),
                 (o_dt + nsb * ldm * 4, o_mv), (o_mv + M * ldus * 4, o_dd),
                 (o_dd + M * nsb * 8, plane.size)):
        assert np.all(plane[a:b] == 0)
    blocks = raw.reshape(M, nsb, 144)
    assert np.array_equal(plane[:M * K // 2].reshape(M, nsb, 128), blocks[:, :, 16:])
    dec = [[orc.q4k_decode_block(blocks[m, b]) for b in range(nsb)] for m in range(M)]
    sc = np.array([[dec[m][b][1] for b in range(nsb)] for m in range(M)]).reshape(M, nc)
    mn = np.array([[dec[m][b][2] for b in range(nsb)] for m in range(M)]).reshape(M, nc)
    d = np.array([[dec[m][b][3] for b in range(nsb)] for m in range(M)])
    dmin = np.array([[dec[m][b][4] for b in range(nsb)] for m in range(M)])
    assert np.array_equal(plane[o_sc:o_sc + M * nc].reshape(M, nc), sc)
    assert np.array_equal(plane[o_mn:o_mn + M * nc].reshape(M, nc), mn)
    dt = plane[o_dt:o_dt + nsb * ldm * 4].view(np.float32).reshape(nsb, ldm)
    assert np.array_equal(dt[:, :M].astype(np.float64), d.T) and np.all(dt[:, M:] == 0)
    mv = plane[o_mv:o_mv + M * ldus * 4].view(np.float32).reshape(M, ldus)
    mv_exact = np.repeat(dmin, 8, axis=1) * mn            # dmin * m in double (exact)
    assert np.array_equal(mv, tf32_pairs(mv_exact.astype(np.float32)))
    pairs = mv[:, :16 * nsb].reshape(M, nsb, 2, 8).astype(np.float64)
    assert np.array_equal((pairs[:, :, 0] + pairs[:, :, 1]).reshape(M, nc), mv_exact)
    ddm = plane[o_dd:o_dd + M * nsb * 8].view(np.float32).reshape(M, nsb, 2)
    assert np.array_equal(ddm[:, :, 0].astype(np.float64), d)
    assert np.array_equal(ddm[:, :, 1].astype(np.float64), dmin)
    codes = np.stack([np.concatenate([dec[m][b][0] for b in range(nsb)]) for m in range(M)])
    assert np.array_equal(host(w.wq).astype(np.int64),
                          np.repeat(sc, 32, axis=1) * codes.astype(np.int64))
    assert np.array_equal(host(q6.q4k_unpack_weights(w)), host(w.wq))
    # the same planes from host memory
    import torch
    wh = q6.q4k_pack_weights(torch.from_numpy(raw), M, K, wq=True)
    assert torch.equal(wh.plane, w.plane) and torch.equal(wh.wq, w.wq)


def q4k_path(N, source):
    """The path a q4_K call with Xq takes: the few-token kernels for N <= 16,
    and on token groups of at most 32 for up to 32 tokens on either source and
    up to 64 tokens from the packed plane."""
    import q6_int8_mmq_gb300 as q6mod
    if N <= q6mod.Q4K_SKINNY_MAX_N or N <= q6mod.Q4K_GROUP_N or (
            source == "raw" and N <= q6mod.Q4K_GROUPS_MAX_N):
        return "q4k_skinny"
    return {"raw": "q4k_tc_raw", "wq": "q4k_tc_wq"}[source]


Q4_SHAPES = [(64, 256, 1), (256, 512, 8), (130, 1024, 3), (300, 768, 12), (300, 768, 16),
             (1001, 2816, 5),
             (1, 256, 3), (7, 2304, 9),   # one row; 9 super-blocks: a stage of one
             (5000, 256, 4),              # more row units than SMs
             (77, 4352, 31),              # the 17-32-token form, 17 super-blocks
             (130, 1024, 17), (200, 768, 129), (384, 768, 300),
             (1016, 768, 2555),    # the split last round of tiles, ragged band and tile
             (1016, 512, 2555),    # split halves of one super-block each (one min pair group)
             (3001, 512, 40), (500, 1024, 48), (500, 1024, 49),
             (300, 2304, 64), (500, 1024, 65),   # groups of 32 + 32; past the groups
             (4800, 768, 12), (4800, 768, 24),   # 32-row units in both MMA forms
             (1000, 1280, 20)]                   # 17-32 form: a last stage of one


@pytest.mark.parametrize("source", ["raw", "wq"])
@pytest.mark.parametrize("M,K,N", Q4_SHAPES, ids=lambda v: str(v))
def test_q4k_mmq_small(q6, orc, M, K, N, source):
    raw = synth.q4k_raw_weights(0x51361201 + M + N, M, K)
    X = synth.activations(0x51361202 + M + N, N, K, outlier_frac=0.02)
    w = q6.q4k_pack_weights(dev(raw), M, K, wq=source == "wq")
    act, xq_o, da_o = quantize(q6, orc, X)
    Y, path, P = q6.q4k_mmq(w, act, source=source, partials=True)
    q6.sync_status()
    assert path == q4k_path(N, source)
    want_p = N * M * K // 32 <= 40_000_000
    if want_p:
        Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
        assert np.array_equal(host(P), Po), "sub-block partials differ"
    else:
        Yo = orc.q4k_mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"q4k {M}x{K}x{N} {source}")
    Y2, _, _ = q6.q4k_mmq(w, act, source=source)
    q6.sync_status()
    check_y(host(Y2), Yo, f"q4k {M}x{K}x{N} {source} fast")


def _q4k_sweep_shapes(count=12, seed=0x5EED4):
    """Seeded irregular shapes: ragged M and N, 1..24 super-blocks per row,
    token counts from one to several rounds of tiles (some with the split
    last round)."""
    rng = np.random.default_rng(seed)
    shapes = []
    for i in range(count):
        N = int([rng.integers(1, 17), rng.integers(17, 700), rng.integers(700, 2700)][i % 3])
        M = int(rng.integers(1, 3000))
        K = 256 * int(rng.integers(1, 25))
        shapes.append((M, K, N))
    return shapes


@pytest.mark.parametrize("M,K,N", _q4k_sweep_shapes(), ids=lambda v: str(v))
def test_q4k_seeded_shape_sweep(q6, orc, M, K, N):
    """Y within tolerance on every output of seeded irregular shapes (from
    the packed plane), and bit-exact sub-block partials where they stay
    small."""
    raw = synth.q4k_raw_weights(0x51361501 + M + K + N, M, K)
    X = synth.activations(0x51361502 + M + K + N, N, K, outlier_frac=0.01)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    act, xq_o, da_o = quantize(q6, orc, X)
    want_p = N * M * (K // 32) <= 20_000_000
    Y, path, P = q6.q4k_mmq(w, act, source="raw", partials=want_p)
    q6.sync_status()
    assert path == q4k_path(N, "raw")
    if want_p:
        Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
        assert np.array_equal(host(P), Po), "sub-block partials differ"
    else:
        Yo = orc.q4k_mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"q4k sweep {M}x{K}x{N}")


def test_q4k_degenerate(q6, orc):
    """All nibbles 0 leave only the min term; dmin = 0 leaves only the scale
    term; d = dmin = 0 gives Y = 0."""
    M, K, N = 128, 512, 130
    X = synth.activations(0x51361301, N, K)
    act, xq_o, da_o = quantize(q6, orc, X)
    base = synth.q4k_raw_weights(0x51361302, M, K).reshape(-1, 144)
    for label, edit in (("nibbles 0", lambda r: r[:, 16:].fill(0)),
                        ("dmin 0", lambda r: r[:, 2:4].fill(0)),
                        ("d and dmin 0", lambda r: r[:, 0:4].fill(0))):
        raw = base.copy()
        edit(raw)
        raw = raw.reshape(M, -1)
        w = q6.q4k_pack_weights(dev(raw), M, K)
        Y, _, _ = q6.q4k_mmq(w, act)
        q6.sync_status()
        Yo = orc.q4k_mmq(raw, M, K, xq_o, da_o)
        if label == "d and dmin 0":
            assert np.all(host(Y) == 0.0)
        check_y(host(Y), Yo, label)


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 9, 16, 17, 24, 32, 50])
def test_q4k_few_tokens_full(q6, orc, N):
    """The few-token kernels on q4_K weights of the ffn_down shape (dp4a for
    one and two tokens, the f16 MMA kernel for 3-16, its 17-32-token form,
    token groups of 32 beyond): every output within tolerance and every
    sub-block partial P bit-exact."""
    _, _, cfg = synth.workload("ffn_down")
    M, K = cfg["M"], cfg["K"]
    raw = synth.q4k_raw_weights(0x51361601, M, K)
    X = synth.activations(0x51361602 + N, N, K, outlier_frac=0.01)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    act, xq_o, da_o = quantize(q6, orc, X)
    Y, path, P = q6.q4k_mmq(w, act, partials=True)
    q6.sync_status()
    assert path == "q4k_skinny"
    Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
    assert np.array_equal(host(P), Po), "sub-block partials differ"
    check_y(host(Y), Yo, f"q4k few tokens N={N}")
    Y2, _, _ = q6.q4k_mmq(w, act)
    q6.sync_status()
    check_y(host(Y2), Yo, f"q4k few tokens N={N} fast")


def test_q4k_pages_ffn_up_full(q6, orc):
    """The pages' model is q4_k_m: its FFN up projection (18944 x 3584) in
    q4_K against the 3325-token prefill stream, every output within
    tolerance of the oracle, from the resident operand plane."""
    raw, X, cfg = synth.q4k_workload("pages_ffn_up")
    M, K = cfg["M"], cfg["K"]
    w = q6.q4k_pack_weights(dev(raw), M, K, wq=True)
    act, xq_o, da_o = quantize(q6, orc, X)
    Y, path, _ = q6.q4k_mmq(w, act, source="wq")
    q6.sync_status()
    assert path == "q4k_tc_wq"
    check_y(host(Y), orc.q4k_mmq_all(raw, M, K, xq_o, da_o), "q4k pages ffn_up")


def test_q4k_ffn_down_full(q6, orc):
    """q4_K weights of the ffn_down shape (4096 x 11008) against its 3314-token
    activation stream: every output within tolerance of the oracle (run over
    disjoint weight-row ranges on the host cores), from the packed plane and
    from the resident operand plane."""
    _, X, cfg = synth.workload("ffn_down")
    M, K = cfg["M"], cfg["K"]
    raw = synth.q4k_raw_weights(0x51361401, M, K)
    w = q6.q4k_pack_weights(dev(raw), M, K, wq=True)
    act, xq_o, da_o = quantize(q6, orc, X)
    Yo = orc.q4k_mmq_all(raw, M, K, xq_o, da_o)
    for source in ("raw", "wq"):
        Y, _, _ = q6.q4k_mmq(w, act, source=source)
        q6.sync_status()
        check_y(host(Y), Yo, f"q4k ffn_down {source}")


@pytest.mark.parametrize("N", [1, 3, 9, 16, 24, 49])
def test_q4k_extremes_every_path(q6, orc, N):
    """Every q4_K kernel at its largest magnitudes: every nibble 15, sc = m =
    63 (all 12 scale bytes 0xFF), d and dmin 1, every activation code +-127
    (rows of +-1; one row mixed). P = +-15 * 127 * 32 and sc * P reach their
    bounds, and the f16 few-token kernel's binary16 subnormal operands and
    power-of-two-scaled sums their largest values; a second half of the blocks
    has nibbles 0 (only the min term) for contrast. The partials are compared
    bit for bit with the oracle's on the dp4a (N = 1), f16 (3, 9, 16), token
    group (24, from the packed plane) and tensor-core (49) paths."""
    M, K = 96, 768
    nblk = M * (K // 256)
    blocks = np.zeros((nblk, 144), np.uint8)
    blocks[:, 0:4] = [0x00, 0x3C, 0x00, 0x3C]       # d = dmin = 1.0
    blocks[:, 4:16] = 0xFF                           # sc = m = 63 for all 8 sub-blocks
    blocks[:, 16:] = np.where((np.arange(nblk) % 2 == 0)[:, None], 0xFF, 0x00)
    raw = blocks.reshape(M, -1)
    dec = orc.q4k_decode_block(blocks[0])
    assert np.all(dec[0] == 15) and np.all(dec[1] == 63) and np.all(dec[2] == 63)
    X = np.ones((N, K), np.float32)
    X[1::2] *= -1.0                                  # +-1 rows: xq = +-127
    X[0, 256:] = np.where(np.arange(K - 256) % 3 == 0, -1.0, 1.0)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    act, xq_o, da_o = quantize(q6, orc, X)
    assert np.abs(xq_o).min() == 127
    Y, path, P = q6.q4k_mmq(w, act, source="raw", partials=True)
    q6.sync_status()
    assert path == q4k_path(N, "raw")
    Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
    assert np.abs(Po).max() == 15 * 127 * 32             # the bound is reached
    assert np.array_equal(host(P), Po), "sub-block partials differ"
    check_y(host(Y), Yo, f"q4k extremes N={N}")


@pytest.mark.parametrize("N", [1, 2, 5, 16, 20, 40])
def test_q4k_long_rows(q6, orc, N):
    """Rows of K = 65,536 (256 super-blocks: 32 stages of the f16 few-token
    kernel's 3-slot ring, its barrier phases wrapping many times) through the
    dp4a (1, 2), f16 (5, 16), its 17-32-token form (20) and tensor-core (40,
    resident plane) paths: bit-exact partials and Y within tolerance; without
    the debug outputs the same Y bit for bit (two tokens: the kernel with the
    activations staged in shared memory)."""
    import torch
    M, K = 130, 65536
    raw = synth.q4k_raw_weights(0x51361701 + N, M, K)
    X = synth.activations(0x51361702 + N, N, K, outlier_frac=0.01)
    w = q6.q4k_pack_weights(dev(raw), M, K, wq=N == 40)
    act, xq_o, da_o = quantize(q6, orc, X)
    source = "wq" if N == 40 else "raw"
    Y, path, P = q6.q4k_mmq(w, act, source=source, partials=True)
    q6.sync_status()
    assert path == q4k_path(N, source)
    Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
    assert np.array_equal(host(P), Po), "sub-block partials differ"
    check_y(host(Y), Yo, f"q4k long rows N={N}")
    Y2, _, _ = q6.q4k_mmq(w, act, source=source)
    q6.sync_status()
    if N <= q6.Q4K_DP4A_MAX_N:
        assert torch.equal(Y, Y2)
    check_y(host(Y2), Yo, f"q4k long rows N={N} fast")


@pytest.mark.parametrize("K", [92928, 93184])
def test_q4k_two_tokens_staged_and_past_its_shared_memory(q6, orc, K):
    """Two tokens on the kernel that stages the activations in shared memory
    (the largest K it holds, 92,928) and, one super-block beyond, on the
    plain dp4a kernel: Y bit for bit that of the debug run (the plain kernel
    with the partials), and within tolerance of the oracle; as the last group
    of 34 tokens too."""
    import torch
    M = 96
    raw = synth.q4k_raw_weights(0x51361711 + K, M, K)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    for N in (2, 34):
        X = synth.activations(0x51361712 + K + N, N, K, outlier_frac=0.01)
        act, xq_o, da_o = quantize(q6, orc, X)
        Y, path, P = q6.q4k_mmq(w, act, partials=True)
        Y2, path2, _ = q6.q4k_mmq(w, act)
        q6.sync_status()
        assert path == path2 == "q4k_skinny"
        assert torch.equal(Y, Y2)
        Yo, Po = orc.q4k_mmq(raw, M, K, xq_o, da_o, partials=True)
        assert np.array_equal(host(P), Po)
        check_y(host(Y2), Yo, f"q4k two tokens K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(4096, 11008, 1), (4096, 11008, 2), (1, 256, 1),
                                   (131, 2816, 2), (5003, 768, 2), (2059, 1024, 1)],
                         ids=lambda v: str(v))
def test_q4k_mmq_f32_equals_two_calls(q6, orc, M, K, N):
    """The fused one/two-token q4_K call gives bit for bit the Y of
    quantize_act (with block sums) followed by q4k_mmq (the same codes,
    scales, block sums, dot products and order), on ordinary activations and
    on blocks at and beside rounding ties, with subnormal and very large
    scales; Y within tolerance of the oracle on every output. The shapes
    cover the full-size weights, one row, an odd super-block count, more rows
    than warps and one super-block per row."""
    import torch
    from test_gpu_parity import hard_activations
    raw = synth.q4k_raw_weights(0x51361801 + M + N, M, K)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    X0 = synth.activations(0x51361802 + K + N, N, K, outlier_frac=0.01)
    for X in (X0, hard_activations(0x51361803 + N, N, K, big=np.float32(1e30))):
        Xd = dev(X)
        Y, path = q6.q4k_mmq_f32(w, Xd)
        act = q6.quantize_act(Xd, want_us=True)
        Y2, path2, _ = q6.q4k_mmq(w, act)
        q6.sync_status()
        assert path == "q4k_skinny_fused" and path2 == "q4k_skinny"
        assert torch.equal(Y, Y2), "fused and separate quantisation disagree"
    act, xq_o, da_o = quantize(q6, orc, X0)
    Yo = (orc.q4k_mmq_all(raw, M, K, xq_o, da_o) if M * K > 1 << 22
          else orc.q4k_mmq(raw, M, K, xq_o, da_o))
    Y, _ = q6.q4k_mmq_f32(w, dev(X0))
    q6.sync_status()
    check_y(host(Y), Yo, f"q4k fused {M}x{K}x{N}")


@pytest.mark.parametrize("K,N", [(92928, 2), (185856, 1)], ids=lambda v: str(v))
def test_q4k_mmq_f32_largest_k(q6, orc, K, N):
    """The largest K whose codes, scales and block sums fit the fused
    kernel's shared memory for N tokens (232,320 of 232,448 bytes): the same
    Y as the two calls, within tolerance of the oracle; one more super-block
    is refused."""
    import torch
    M = 64
    raw = synth.q4k_raw_weights(0x51361811 + N, M, K)
    X = synth.activations(0x51361812 + N, N, K, outlier_frac=0.01)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    Xd = dev(X)
    Y, path = q6.q4k_mmq_f32(w, Xd)
    act, xq_o, da_o = quantize(q6, orc, X)
    Y2, _, _ = q6.q4k_mmq(w, act)
    q6.sync_status()
    assert path == "q4k_skinny_fused" and torch.equal(Y, Y2)
    check_y(host(Y), orc.q4k_mmq(raw, M, K, xq_o, da_o), f"q4k fused K={K} N={N}")
    K2 = K + 256
    w2 = q6.q4k_pack_weights(dev(synth.q4k_raw_weights(0x51361813, M, K2)), M, K2)
    with pytest.raises(q6.Q6Error):
        q6.q4k_mmq_f32(w2, dev(synth.activations(0x51361814, N, K2)))


def test_q4k_mmq_f32_strided_input_and_output(q6):
    """X with a wider row stride, Y with an odd row stride at an unaligned
    address: the floats between Y's rows stay untouched, the result equals
    the two calls'; three tokens are refused."""
    import torch
    M, K, N = 328, 1024, 2
    raw = synth.q4k_raw_weights(0x51361821, M, K)
    w = q6.q4k_pack_weights(dev(raw), M, K)
    big = torch.full((N, K + 64), float("nan"), dtype=torch.float32, device="cuda")
    big[:, :K] = dev(synth.activations(0x51361822, N, K))
    Xv = big[:, :K]
    ldy = M + 37
    buf = torch.full((N * ldy + 1,), float("nan"), dtype=torch.float32, device="cuda")
    Yv = buf[1:].view(N, ldy)[:, :M]
    Y, path = q6.q4k_mmq_f32(w, Xv, Y=Yv)
    Y2, _, _ = q6.q4k_mmq(w, q6.quantize_act(Xv, want_us=True))
    q6.sync_status()
    assert path == "q4k_skinny_fused" and Y.data_ptr() == Yv.data_ptr()
    assert torch.equal(Yv, Y2)
    b = host(buf)
    assert np.isnan(b[0]) and np.all(np.isnan(b[1:].reshape(N, ldy)[:, M:]))
    with pytest.raises(q6.Q6Error):
        q6.q4k_mmq_f32(w, dev(synth.activations(0x51361823, 3, K)))   # three tokens
