"""q6k_mmq_noalloc agrees with q6k_mmq (needs a GB300).

q6k_mmq_noalloc serves callers that cannot allocate device memory when they
call the GEMM (a fixed budget or pool that forbids new allocations, or a
latency-critical path that must not enter the allocator): its scratch is a
static device array of the library instead of a caller workspace. This test
calls it through the C ABI twice in a row and checks each result against
q6k_mmq on the same inputs and against the CPU oracle, within the GEMM
tolerance of the parity tests, and reads the entry point's own status word
(q6k_mmq_noalloc_status) after each call, so a bounded wait that gave up
would fail the test. It lives in its own file, collected last, and builds
what it needs, so it runs the same alone in a fresh process and after the
other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def close(Y, Yref):
    Y = Y.detach().cpu().numpy().astype(np.float64)
    if not isinstance(Yref, np.ndarray):
        Yref = Yref.detach().cpu().numpy()
    Yref = Yref.astype(np.float64)
    err = np.abs(Y - Yref)
    scale = np.abs(Yref).max()
    assert np.all(np.isfinite(Y))
    assert err.max() <= MAX_REL * scale
    assert err.sum() <= NORMWISE * np.abs(Yref).sum()


def noalloc(q6, w, act, use_wexp, stream=None):
    import torch
    lib = q6.load()
    Y = torch.full((act.N, w.M), float("nan"), dtype=torch.float32, device=w.plane.device)
    path = ctypes.c_int(-1)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    rc = lib.q6k_mmq_noalloc(p(w.plane), p(w.wexp if use_wexp else None), w.M, w.K, p(act.xq),
                             p(act.da), p(act.xh), act.N, p(Y), w.M, ctypes.byref(path), s)
    assert rc == q6.Q6_OK, lib.q6_last_error().decode()
    # waits for the stream; Q6_ETIMEOUT if a kernel of the call gave up a wait
    rc = lib.q6k_mmq_noalloc_status(s)
    assert rc == q6.Q6_OK, lib.q6_last_error().decode()
    return Y, q6.PATH_NAMES[path.value]


@pytest.mark.parametrize("N", [300, 40, 20, 8, 2])  # tensor cores, token groups, 17-24 form, few tokens, two staged
def test_noalloc_matches_q6k_mmq_on_two_calls(q6, N):
    import torch
    M, K = 4096, 4096                     # the largest layer its static scratch holds
    raw = synth.q6k_raw_weights(0x51360777, M, K)
    X = synth.activations(0x51360778, N, K)
    w = q6.pack_weights(torch.from_numpy(raw).cuda(), M, K, wexp=True)
    act = q6.quantize_act(torch.from_numpy(X).cuda())
    orc = oracle.get()
    xq_o, da_o = orc.quantize(X)
    assert np.array_equal(act.xq.cpu().numpy(), xq_o)
    Yo = orc.mmq_all(raw, M, K, xq_o, da_o)
    for use_wexp in (False, True):
        Yref, ref_path, _ = q6.mmq(w, act, source="wexp" if use_wexp else "raw")
        q6.sync_status()
        for _ in range(2):                # two calls in a row share the static scratch
            Y, path = noalloc(q6, w, act, use_wexp)
            assert path == ref_path
            close(Y, Yref)
            close(Y, Yo)


def test_noalloc_rejects_layers_beyond_its_scratch(q6):
    lib = q6.load()
    fake = ctypes.c_void_p(0x10000)       # rejected on the host before any use
    path = ctypes.c_int(-1)
    # 97 tokens: past the token groups, so the unpack and its scratch apply
    rc = lib.q6k_mmq_noalloc(fake, None, 4096, 11008, fake, fake, fake, 97, fake, 4096,
                             ctypes.byref(path), None)
    assert rc == q6.Q6_ESIZE
    assert b"static scratch" in lib.q6_last_error()
    # without Xq, 40 tokens cannot run the token groups either
    rc = lib.q6k_mmq_noalloc(fake, None, 4096, 11008, None, fake, fake, 40, fake, 4096,
                             ctypes.byref(path), None)
    assert rc == q6.Q6_ESIZE
    # the few-token path takes the same size limit on M * K as q6k_mmq
    rc = lib.q6k_mmq_noalloc(fake, None, 1 << 20, 1 << 21, fake, fake, None, 4, fake, 1 << 20,
                             ctypes.byref(path), None)
    assert rc == q6.Q6_ESIZE
