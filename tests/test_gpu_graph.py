"""A sequence of W12 GEMMs captured in a CUDA graph and replayed.

A model's forward pass (or the 64-layer stack of the benchmark) launches one
GEMM per weight tensor; capturing the sequence in a CUDA graph removes the
host launch cost.  Each GEMM here reads the previous one's output, and the
graph is replayed twice with and without W12_GEMM_OVERLAP_PREVIOUS (whose
programmatic-dependent launches become graph edges).  The replays must give
bitwise the same outputs as eager calls, and leave the shared workspace's
arrival counters at zero.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 16, 48])
@pytest.mark.parametrize("flags", [0, 1])
def test_graph_replay_matches_eager_calls(M, flags, w12lib):
    dims = (1024, 3072, 1024, 2048, 768)
    ts = [w12lib.w12_encode(synth.dense_weights_device(dims[i + 1], dims[i], seed=120 + i))
          for i in range(len(dims) - 1)]
    x0 = synth.activations_device(M, dims[0], seed=130 + M)
    outs = [torch.empty(M, d, dtype=torch.bfloat16, device="cuda") for d in dims[1:]]
    ws = w12lib.Workspace("cuda", 1 << 22)
    stream = torch.cuda.Stream()
    opts = w12lib.make_opts(flags=flags)
    calls = []
    x = x0
    for t, y in zip(ts, outs):
        calls.append(w12lib.GemmCall(x, t, y, ws, opts=opts, stream=stream))
        x = y

    with torch.cuda.stream(stream):
        for c in calls:  # eager run (also fills the launch caches before capture)
            c()
    torch.cuda.synchronize()
    eager = [synth.tensor_to_bits(y) for y in outs]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    for _ in range(2):
        for y in outs:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, y in zip(eager, outs):
            assert np.array_equal(a, synth.tensor_to_bits(y))
    assert int(ws.buf[256:256 + 4 * 1024].sum()) == 0
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK
