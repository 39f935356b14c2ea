"""The tensor-core GEMM with the quantiser fused into its producer
(q6k_mmq_f32_tc; needs a GB300).

The fused kernel reads f32 X and forms the binary16 codes and the per-32 scale
da of each block in shared memory with the standalone quantiser's arithmetic,
so its Y must be bit for bit that of q8_quantize_act + q6k_mmq on the
tensor-core path (N > 16), and within the method's tolerance of the oracle
(max|Y - Yo| <= 1e-3 max|Yo|, sum|Y - Yo| / sum|Yo| <= 1e-5) for every N.
This is the pages' r34 prepass turned back into the GEMM ("r38 -- q6_K
BT-style raw-byte mma kernel", Sec. 1).
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


def separate(q6, W, Xd, source):
    act = q6.quantize_act(Xd, want_xq=False)
    Y, path, _ = q6.mmq(W, act, source=source)
    return Y, path


SHAPES = [(256, 512, 130), (300, 768, 257),   # ragged weight band and token tile
          (1016, 768, 2555),                  # the split last round of tiles
          (1016, 512, 2555),                  # split halves of one super-block each
          (4096, 1024, 700), (128, 256, 129)]


@pytest.mark.parametrize("source", ["raw", "wh"])
@pytest.mark.parametrize("M,K,N", SHAPES, ids=lambda v: str(v))
def test_fused_equals_separate_and_oracle(q6, orc, M, K, N, source):
    raw = synth.q6k_raw_weights(0x51362001 + M + N, M, K)
    X = synth.activations(0x51362002 + M + N, N, K, outlier_frac=0.02)
    X[0, :32] = 0.0                       # a zero block: da = 0, codes 0
    X[N // 2, 64:96] *= 1e-30             # tiny scales
    W = q6.pack_weights(dev(raw), M, K, wh=source == "wh")
    Xd = dev(X)
    Y, path = q6.mmq_f32_tc(W, Xd, source=source)
    q6.sync_status()
    assert path == {"raw": "tc_fused_raw", "wh": "tc_fused_wh"}[source]
    Ys, spath = separate(q6, W, Xd, source)
    q6.sync_status()
    assert spath.startswith("tc_")
    import torch
    assert torch.equal(Y, Ys), "fused quantiser differs from quantize_act + mmq"
    xq_o, da_o = orc.quantize(X)
    small = N * M * K <= 1 << 30
    Yo = orc.mmq(raw, M, K, xq_o, da_o) if small else orc.mmq_all(raw, M, K, xq_o, da_o)
    check_y(host(Y), Yo, f"fused {M}x{K}x{N} {source}")


def _fused_sweep_shapes(count=8, seed=0x5EEDF):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 3000)), 256 * int(rng.integers(1, 25)),
             int(rng.integers(17, 2700))) for _ in range(count)]


@pytest.mark.parametrize("M,K,N", _fused_sweep_shapes(), ids=lambda v: str(v))
def test_fused_seeded_shape_sweep(q6, orc, M, K, N):
    """Seeded irregular shapes: bit for bit the separate path, and within
    tolerance of the oracle."""
    import torch
    raw = synth.q6k_raw_weights(0x51362301 + M + K + N, M, K)
    X = synth.activations(0x51362302 + M + K + N, N, K, outlier_frac=0.01)
    W = q6.pack_weights(dev(raw), M, K)
    Xd = dev(X)
    Y, _ = q6.mmq_f32_tc(W, Xd, source="raw")
    Ys, _ = separate(q6, W, Xd, "raw")
    q6.sync_status()
    assert torch.equal(Y, Ys)
    xq_o, da_o = orc.quantize(X)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), f"fused sweep {M}x{K}x{N}")


@pytest.mark.parametrize("N", [1, 5, 16])
def test_fused_few_tokens_against_oracle(q6, orc, N):
    """Small N runs the tensor-core kernel with one ragged token tile (the
    separate path would take the few-token kernels, with another summation
    order): checked against the oracle."""
    M, K = 384, 1024
    raw = synth.q6k_raw_weights(0x51362101 + N, M, K)
    X = synth.activations(0x51362102 + N, N, K)
    W = q6.pack_weights(dev(raw), M, K)
    Y, path = q6.mmq_f32_tc(W, dev(X))
    q6.sync_status()
    assert path == "tc_fused_raw"
    xq_o, da_o = orc.quantize(X)
    check_y(host(Y), orc.mmq(raw, M, K, xq_o, da_o), f"fused N={N}")


def test_fused_row_stride(q6):
    """X as a view with ldx > K (rows 16-byte aligned): the same Y as from a
    contiguous copy."""
    import torch
    M, K, N = 256, 768, 200
    raw = synth.q6k_raw_weights(0x51362201, M, K)
    X = synth.activations(0x51362202, N, K + 64)
    W = q6.pack_weights(dev(raw), M, K, wh=True)
    Xw = dev(X)
    Y1, _ = q6.mmq_f32_tc(W, Xw[:, 32:32 + K])
    Y2, _ = q6.mmq_f32_tc(W, Xw[:, 32:32 + K].contiguous())
    q6.sync_status()
    assert torch.equal(Y1, Y2)


def test_fused_ffn_down_full(q6, orc):
    """The ffn_down workload (4096 x 11008, 3314 tokens), in the launch
    configuration the benchmark times: bit for bit the separate path, and
    every output within tolerance of the oracle."""
    import torch
    raw, X, cfg = synth.workload("ffn_down")
    M, K = cfg["M"], cfg["K"]
    W = q6.pack_weights(dev(raw), M, K, wh=True)
    Xd = dev(X)
    Y, path = q6.mmq_f32_tc(W, Xd, source="wh")
    Ys, _ = separate(q6, W, Xd, "wh")
    q6.sync_status()
    assert path == "tc_fused_wh"
    assert torch.equal(Y, Ys)
    xq_o, da_o = orc.quantize(X)
    check_y(host(Y), orc.mmq_all(raw, M, K, xq_o, da_o), "fused ffn_down")
