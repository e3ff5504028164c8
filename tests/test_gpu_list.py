"""w12_gemm_list (several small-M GEMMs in one persistent launch) and the
fused gate/up epilogue W12_GEMM_SILU_MUL.

SpecPilot (arXiv 2611.02501): the exact pass streams every target weight
(section 4.1) and weight reads are 80% of a verify step (English summary,
section 6.1), so a layer pass runs as one chain of W12 GEMMs.  The list call
must give, for every item, bitwise the Y that w12_gemm gives (same cut, same
order), must read an item's activations only after the item it depends on
has written them, and must leave its workspace clean.  The fused epilogue
(reading R24: silu(g) * u of rows 16s+i and 16s+8+i) is checked against the
oracle's FP64 silu(g) * u with the rule in tests/w12_tol.py.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures, silu_mul_tolerance_failures

pytestmark = pytest.mark.gpu


def bits(x):
    return synth.tensor_to_bits(x)


def encode(w12lib, W):
    return w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))


def test_list_equals_w12_gemm_bitwise(w12lib, oracle):
    """Independent items of mixed shapes, M and escape density: every Y is
    the one w12_gemm gives, bit for bit, and within tolerance of the oracle."""
    shapes = [(1024, 3000, 1, "dense"), (2000, 1024, 5, "adversarial"), (4096, 2048, 8, "dense"),
              (77, 264, 3, "adversarial"), (5121, 1536, 16, "dense"), (640, 17400, 12, "dense")]
    entries, refs = [], []
    for i, (N, K, M, kind) in enumerate(shapes):
        W = (synth.dense_weights if kind == "dense" else synth.adversarial_weights)(N, K, seed=100 + i)
        A = synth.activations(M, K, seed=200 + i)
        t = encode(w12lib, W)
        Ad = synth.bits_to_tensor(A, "cuda")
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        entries.append((Ad, t, Y, -1, 0))
        refs.append((W, A, w12lib.w12_gemm(Ad, t)))
    ws = w12lib.Workspace("cuda")
    call = w12lib.GemmListCall(entries, ws)
    for _ in range(2):  # twice: the workspace is left clean and reusable
        call()
        torch.cuda.synchronize()
        for (Ad, t, Y, _, _), (W, A, Yg) in zip(entries, refs):
            assert np.array_equal(bits(Y), bits(Yg))
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK
    for (Ad, t, Y, _, _), (W, A, Yg) in list(zip(entries, refs))[:4]:
        st, ref = oracle.encode(W)
        st, Yr, Y64, mag = oracle.gemm(A, ref)
        assert gemm_tolerance_failures(bits(Y), Yr, Y64, mag).size == 0


def chain_entries(w12lib, M, seed, silu_hidden=None):
    """A chain x -> A (1536 -> 3072) -> B (3072 -> 1024) [-> gate/up (1024 ->
    2H, fused silu) -> down (H -> 1024)]: each item's A is the previous
    item's Y, declared with `after`."""
    dims = [(3072, 1536), (1024, 3072)]
    if silu_hidden:
        dims += [(2 * silu_hidden, 1024), (1024, silu_hidden)]
    x = synth.activations_device(M, 1536, seed=seed)
    entries, tensors = [], []
    A = x
    for i, (N, K) in enumerate(dims):
        t = w12lib.w12_encode(synth.dense_weights_device(N, K, seed=seed + 10 + i))
        flags = w12lib.W12_GEMM_SILU_MUL if (silu_hidden and i == 2) else 0
        cols = N // 2 if flags else N
        Y = torch.full((M, cols), float("nan"), dtype=torch.bfloat16, device="cuda")
        entries.append((A, t, Y, i - 1, flags))
        tensors.append(t)
        A = Y
    return x, entries


@pytest.mark.parametrize("M", [1, 8, 16])
def test_dependent_chain_reads_finished_outputs(M, w12lib):
    """Each item's activations are the previous item's output: the chain's
    results equal w12_gemm called one after another on the same inputs."""
    x, entries = chain_entries(w12lib, M, seed=300 + M, silu_hidden=2048)
    ws = w12lib.Workspace("cuda")
    call = w12lib.GemmListCall(entries, ws)
    for rep in range(3):
        # new inputs each time, so an output read before it was rewritten
        # (a stale copy from the previous call) could not pass
        x.copy_(synth.activations_device(M, 1536, seed=310 + 10 * M + rep))
        for _, _, Y, _, _ in entries:
            Y.fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        A = x
        for (_, t, Y, _, flags) in entries:
            want = w12lib.w12_gemm(A, t, opts=w12lib.make_opts(flags=flags))
            assert np.array_equal(bits(Y), bits(want)), rep
            A = want
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK


@pytest.mark.parametrize("cap", [1, 7, 76, 152, 1000])
def test_list_across_grids(cap, w12lib):
    x, entries = chain_entries(w12lib, 4, seed=400, silu_hidden=1024)
    ws = w12lib.Workspace("cuda")
    w12lib.GemmListCall(entries, ws)()
    torch.cuda.synchronize()
    want = [bits(e[2]).copy() for e in entries]
    w12lib.GemmListCall(entries, ws, w12lib.make_opts(max_ctas=cap))()
    torch.cuda.synchronize()
    for e, wv in zip(entries, want):
        assert np.array_equal(bits(e[2]), wv)


def test_list_longer_than_one_launch(w12lib):
    """70 items (two launches of at most 64): a chain that crosses the
    launch boundary, and independent items."""
    N = K = 512
    ts = [w12lib.w12_encode(synth.dense_weights_device(N, K, seed=500 + i)) for i in range(5)]
    x = synth.activations_device(2, K, seed=501)
    entries, A = [], x
    for i in range(70):
        Y = torch.empty(2, N, dtype=torch.bfloat16, device="cuda")
        after = i - 1 if i % 3 else -1  # chains of three
        entries.append((A if after >= 0 else x, ts[i % 5], Y, after, 0))
        A = Y
    w12lib.w12_gemm_list(entries, w12lib.Workspace("cuda"))
    torch.cuda.synchronize()
    prev = None
    for i, (A, t, Y, after, _) in enumerate(entries):
        src = x if after < 0 else prev
        assert np.array_equal(bits(Y), bits(w12lib.w12_gemm(src, t))), i
        prev = Y


def test_list_edge_items(w12lib):
    """M = 0 and K = 0 items, an item that depends on an empty one."""
    t0 = w12lib.w12_encode(synth.dense_weights_device(256, 0 + 256, seed=600))
    tk0 = w12lib.w12_encode(torch.empty(64, 0, dtype=torch.bfloat16, device="cuda"))
    A = synth.activations_device(3, 256, seed=601)
    Y0 = torch.full((3, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    Ye = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    Y1 = torch.empty(3, 256, dtype=torch.bfloat16, device="cuda")
    entries = [(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), t0, Ye, -1, 0),
               (torch.empty(3, 0, dtype=torch.bfloat16, device="cuda"), tk0, Y0, -1, 0),
               (A, t0, Y1, 0, 0)]
    w12lib.w12_gemm_list(entries, w12lib.Workspace("cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y0) == 0
    assert np.array_equal(bits(Y1), bits(w12lib.w12_gemm(A, t0)))


def test_list_stall_reports_timeout(w12lib):
    """W12_GEMM_TEST_STALL makes the first item's dependency wait run out
    (bounded: about a second); the call completes, the status says
    W12_ERR_TIMEOUT, and the next call is right again."""
    x, entries = chain_entries(w12lib, 2, seed=700)
    ws = w12lib.Workspace("cuda")
    w12lib.GemmListCall(entries, ws, w12lib.make_opts(flags=w12lib.W12_GEMM_TEST_STALL))()
    torch.cuda.synchronize()
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_ERR_TIMEOUT
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK
    w12lib.GemmListCall(entries, ws)()
    torch.cuda.synchronize()
    A = x
    for (_, t, Y, _, _) in entries:
        want = w12lib.w12_gemm(A, t)
        assert np.array_equal(bits(Y), bits(want))
        A = want


def test_list_rejects_bad_items(w12lib):
    t = w12lib.w12_encode(synth.dense_weights_device(64, 256, seed=800))
    A = synth.activations_device(4, 256, seed=801)
    Y = torch.empty(4, 64, dtype=torch.bfloat16, device="cuda")
    ws = w12lib.Workspace("cuda")
    with pytest.raises(ValueError):
        w12lib.GemmListCall([(A, t, Y, 0, 0)], ws)  # depends on itself
    A17 = synth.activations_device(17, 256, seed=802)
    Y17 = torch.empty(17, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w12lib.W12Error):
        w12lib.GemmListCall([(A17, t, Y17, -1, 0)], ws)()  # M > 16: the list is the small-M path


# ---- the fused gate/up epilogue ----

@pytest.mark.parametrize("M", [1, 5, 16, 24, 33, 64, 130])
def test_silu_mul_against_the_oracle(M, w12lib, oracle):
    """Gate/up rows interleaved per stripe (8 gate rows, then their 8 up
    rows); both GEMM paths, several splits."""
    N, K = 2 * 1536, 2048
    W = synth.dense_weights(N, K, seed=900 + M)
    A = synth.activations(M, K, seed=910 + M)
    st, ref = oracle.encode(W)
    st, Yr, g, u, mg, mu = oracle.gemm_silu_mul(A, ref)
    assert st == oracle.OK
    t = encode(w12lib, W)
    Ad = synth.bits_to_tensor(A, "cuda")
    for split in (0, 1, 3):
        Y = w12lib.w12_gemm(Ad, t, opts=w12lib.make_opts(split_k=split, flags=w12lib.W12_GEMM_SILU_MUL))
        torch.cuda.synchronize()
        assert tuple(Y.shape) == (M, N // 2)
        bad = silu_mul_tolerance_failures(bits(Y), Yr, g, u, mg, mu)
        assert bad.size == 0, (split, bad[:8])


def test_silu_mul_balanced_ranges(w12lib, oracle):
    """M > 128 on a large layer takes the balanced-range kernel."""
    N, K, M = 9728, 8192, 136
    W = synth.dense_weights(N, K, seed=920)
    A = synth.activations(M, K, seed=921)
    t = encode(w12lib, W)
    Ad = synth.bits_to_tensor(A, "cuda")
    Y = bits(w12lib.w12_gemm(Ad, t, opts=w12lib.make_opts(flags=w12lib.W12_GEMM_SILU_MUL)))
    rows = np.arange(0, N, 16 * 37)[:16]  # sampled stripes: both rows of each hidden unit
    sub = np.concatenate([np.arange(r, r + 16) for r in rows])
    st, ref = oracle.encode(W[sub])
    st, Yr, g, u, mg, mu = oracle.gemm_silu_mul(A, ref)
    cols = np.concatenate([np.arange(r // 2, r // 2 + 8) for r in rows])
    assert silu_mul_tolerance_failures(Y[:, cols], Yr, g, u, mg, mu).size == 0


def test_silu_mul_matches_plain_gemm_then_silu(w12lib):
    """On the small-M path the fused result is the plain GEMM's FP32 sums
    passed through silu: the same value as silu applied in FP32 to the
    unrounded sums, so it is checked against the plain GEMM within one BF16
    rounding of each operand."""
    N, K, M = 512, 1024, 4
    t = w12lib.w12_encode(synth.dense_weights_device(N, K, seed=930))
    A = synth.activations_device(M, K, seed=931)
    Y = w12lib.w12_gemm(A, t, opts=w12lib.make_opts(flags=w12lib.W12_GEMM_SILU_MUL)).float()
    P = w12lib.w12_gemm(A, t).float().view(M, N // 16, 2, 8)
    g, u = P[:, :, 0, :].reshape(M, -1), P[:, :, 1, :].reshape(M, -1)
    approx = torch.nn.functional.silu(g) * u
    assert torch.allclose(Y, approx, rtol=3e-2, atol=1e-2)


def test_silu_mul_rejects_bad_n(w12lib):
    t = w12lib.w12_encode(synth.dense_weights_device(40, 256, seed=940))
    A = synth.activations_device(2, 256, seed=941)
    with pytest.raises(ValueError):
        w12lib.w12_gemm(A, t, opts=w12lib.make_opts(flags=w12lib.W12_GEMM_SILU_MUL))
