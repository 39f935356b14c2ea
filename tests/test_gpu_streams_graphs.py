"""The C ABI on a caller's stream and inside a CUDA graph (needs a GB300).

Every call is asynchronous on the stream it is given and allocates nothing on
the hot path, so the whole per-batch path (quantise, unpack, GEMM) can run on
a side stream and can be captured once into a CUDA graph and replayed with new
inputs. Results are checked against the oracle with the GEMM tolerance.
"""
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


def close(Y, Yo):
    Y = Y.detach().cpu().numpy().astype(np.float64)
    err = np.abs(Y - Yo)
    assert np.all(np.isfinite(Y))
    assert err.max() <= MAX_REL * np.abs(Yo).max()
    assert err.sum() <= NORMWISE * np.abs(Yo).sum()


def expected(raw, M, K, X):
    orc = oracle.get()
    xq, da = orc.quantize(X)
    return orc.mmq(raw, M, K, xq, da)


@pytest.mark.parametrize("N", [200, 9])   # tensor-core and skinny kernels
def test_path_on_a_side_stream(q6, N):
    import torch
    M, K = 256, 768
    raw = synth.q6k_raw_weights(0x51360901, M, K)
    X = synth.activations(0x51360902 + N, N, K)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        w = q6.pack_weights(torch.from_numpy(raw).cuda(), M, K, stream=side)
        act = q6.quantize_act(torch.from_numpy(X).cuda(), stream=side)
        Y, path, _ = q6.mmq(w, act, source="raw", stream=side)
    q6.sync_status(side)
    assert path == ("skinny" if N <= q6.SKINNY_MAX_N else "tc_raw")
    close(Y, expected(raw, M, K, X))


def test_whole_path_in_a_cuda_graph(q6):
    """quantise + unpack + GEMM captured once, replayed for two inputs."""
    import torch
    M, K, N = 384, 1024, 300
    raw = synth.q6k_raw_weights(0x51360903, M, K)
    X1 = synth.activations(0x51360904, N, K)
    X2 = synth.activations(0x51360905, N, K, outlier_frac=0.02)
    w = q6.pack_weights(torch.from_numpy(raw).cuda(), M, K)
    Xs = torch.from_numpy(X1).cuda()             # static input of the graph
    act = q6.alloc_activations(N, K)
    Y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    ws = torch.empty(q6.workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")

    def step():
        q6.quantize_act(Xs, out=act)
        q6.mmq(w, act, Y=Y, source="raw", workspace=ws)

    step()                                       # first use of the device: set-up runs here
    q6.sync_status()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    for X in (X1, X2):
        Xs.copy_(torch.from_numpy(X).cuda())
        Y.fill_(float("nan"))
        graph.replay()
        q6.sync_status()
        close(Y, expected(raw, M, K, X))


@pytest.mark.parametrize("N", [1, 2])
def test_fused_call_on_a_side_stream_and_in_a_graph(q6, N):
    """q6k_mmq_f32 (quantiser and GEMM in one kernel) on a caller's side
    stream, then captured into a CUDA graph and replayed for two inputs."""
    import torch
    M, K = 512, 2048
    raw = synth.q6k_raw_weights(0x51360911 + N, M, K)
    X1 = synth.activations(0x51360912 + N, N, K)
    X2 = synth.activations(0x51360913 + N, N, K, outlier_frac=0.02)
    w = q6.pack_weights(torch.from_numpy(raw).cuda(), M, K)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        Y, path = q6.mmq_f32(w, torch.from_numpy(X1).cuda(), stream=side)
    q6.sync_status(side)
    assert path == "skinny_fused"
    close(Y, expected(raw, M, K, X1))
    Xs = torch.from_numpy(X1).cuda()             # static input of the graph
    Ys = torch.empty((N, M), dtype=torch.float32, device="cuda")
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            q6.mmq_f32(w, Xs, Y=Ys)
    for X in (X1, X2):
        Xs.copy_(torch.from_numpy(X).cuda())
        Ys.fill_(float("nan"))
        graph.replay()
        q6.sync_status()
        close(Ys, expected(raw, M, K, X))


@pytest.mark.parametrize("N,source", [(1, "raw"), (6, "raw"), (16, "raw"), (30, "raw"),
                                      (30, "wq"), (200, "raw")])
def test_q4k_path_in_a_cuda_graph(q6, N, source):
    """The q4_K step (quantiser with block sums, then q4k_mmq) captured once
    into a CUDA graph and replayed for two inputs, on every path: dp4a (1),
    the f16 few-token kernel (6, 16), its token groups (30 from the packed
    plane), the tensor cores with K split (30 on the resident plane) and the
    unpack + tensor cores (200). The few-token kernels start as dependent
    launches of the quantiser inside the graph."""
    import torch
    M, K = 300, 1536
    raw = synth.q4k_raw_weights(0x51360921 + N, M, K)
    X1 = synth.activations(0x51360922 + N, N, K)
    X2 = synth.activations(0x51360923 + N, N, K, outlier_frac=0.02)
    w = q6.q4k_pack_weights(torch.from_numpy(raw).cuda(), M, K, wq=source == "wq")
    Xs = torch.from_numpy(X1).cuda()             # static input of the graph
    act = q6.alloc_activations(N, K, want_us=True)
    Y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    ws = torch.empty(4 * M * K + (1 << 22), dtype=torch.uint8, device="cuda")
    path = [None]

    def step():
        q6.quantize_act(Xs, out=act)
        path[0] = q6.q4k_mmq(w, act, Y=Y, source=source, workspace=ws)[1]

    step()
    q6.sync_status()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    orc = oracle.get()
    for X in (X1, X2):
        Xs.copy_(torch.from_numpy(X).cuda())
        Y.fill_(float("nan"))
        graph.replay()
        q6.sync_status()
        xq, da = orc.quantize(X)
        close(Y, orc.q4k_mmq(raw, M, K, xq, da))
    assert path[0] == ("q4k_skinny" if N <= q6.Q4K_GROUP_N or
                       (source == "raw" and N <= q6.Q4K_GROUPS_MAX_N) else
                       {"raw": "q4k_tc_raw", "wq": "q4k_tc_wq"}[source])


@pytest.mark.parametrize("N", [1, 2])
def test_q4k_fused_call_on_a_side_stream_and_in_a_graph(q6, N):
    """q4k_mmq_f32 (quantiser with block sums and the q4_K GEMM in one
    kernel) on a caller's side stream, then two such calls chained in one
    CUDA graph, the second reading the first's Y as its activations (a
    dependent launch that must see the previous kernel's writes), replayed
    for two inputs."""
    import torch
    orc = oracle.get()
    M1, K1, M2 = 512, 2048, 768             # layer 2 takes layer 1's 512 outputs
    raw1 = synth.q4k_raw_weights(0x51360931 + N, M1, K1)
    raw2 = synth.q4k_raw_weights(0x51360932 + N, M2, M1)
    X1 = synth.activations(0x51360933 + N, N, K1)
    X2 = synth.activations(0x51360934 + N, N, K1, outlier_frac=0.02)
    w1 = q6.q4k_pack_weights(torch.from_numpy(raw1).cuda(), M1, K1)
    w2 = q6.q4k_pack_weights(torch.from_numpy(raw2).cuda(), M2, M1)

    def expect(raw, M, K, X):
        xq, da = orc.quantize(X)
        return orc.q4k_mmq(raw, M, K, xq, da)

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        Y, path = q6.q4k_mmq_f32(w1, torch.from_numpy(X1).cuda(), stream=side)
    q6.sync_status(side)
    assert path == "q4k_skinny_fused"
    close(Y, expect(raw1, M1, K1, X1))
    Xs = torch.from_numpy(X1).cuda()             # static input of the graph
    Y1 = torch.empty((N, M1), dtype=torch.float32, device="cuda")
    Y2 = torch.empty((N, M2), dtype=torch.float32, device="cuda")
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            q6.q4k_mmq_f32(w1, Xs, Y=Y1)
            q6.q4k_mmq_f32(w2, Y1, Y=Y2)
    for X in (X1, X2):
        Xs.copy_(torch.from_numpy(X).cuda())
        Y1.fill_(float("nan"))
        Y2.fill_(float("nan"))
        graph.replay()
        q6.sync_status()
        y1 = Y1.cpu().numpy()
        close(Y1, expect(raw1, M1, K1, X))
        # layer 2 against the oracle on the GPU's own layer-1 output
        close(Y2, expect(raw2, M2, M1, y1))
