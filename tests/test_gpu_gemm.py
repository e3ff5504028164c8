"""GPU W12 GEMM against the oracle, and its determinism.

SpecPilot (arXiv 2611.02501), section 4.1: the GEMM decodes records in
registers and splits the reduction in a fixed order, so it is deterministic.
Parity: every output within 2 BF16 ulp of the oracle's FP64 sum rounded to
BF16, or within 1e-3 * sum|a||w| of the FP64 sum (tests/w12_tol.py);
exact-result cases bitwise; repeated runs and grid sizes bitwise identical.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def run_gpu(w, W, A, opts=None, t=None):
    if t is None:
        t = w.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    Y = w.w12_gemm(Ad, t, opts=opts)
    torch.cuda.synchronize()
    return synth.tensor_to_bits(Y), t


def check_parity(oracle, w, W, A, opts=None):
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    assert st == oracle.OK
    Yg, t = run_gpu(w, W, A, opts)
    bad = gemm_tolerance_failures(Yg, Yr, Y64, mag)
    assert bad.size == 0, (bad[:10], Yg.reshape(-1)[bad[:10]], Yr.reshape(-1)[bad[:10]])
    return Yg, Yr


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 12, 15, 16])
def test_dense_1024(M, w12lib, oracle):
    W = synth.dense_weights(1024, 1024, seed=0)
    A = synth.activations(M, 1024, seed=1000 + M)
    check_parity(oracle, w12lib, W, A)


@pytest.mark.parametrize("N,K,M", [(1, 1, 1), (3, 65, 2), (16, 64, 1), (77, 1000, 5), (40, 17400, 8),
                                   (130, 257, 16), (333, 600, 11), (17, 1, 3)])
def test_ragged_shapes(N, K, M, w12lib, oracle):
    Kpad = (K + 7) // 8 * 8
    W = synth.dense_weights(N, K, seed=N * 7 + K)
    A = np.zeros((M, Kpad), np.uint16)
    A[:, :K] = synth.activations(M, K, seed=K)
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(np.ascontiguousarray(A[:, :K]), ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")[:, :K]  # row stride Kpad (a multiple of 8)
    Y = w12lib.w12_gemm(Ad, t)
    Yg = synth.tensor_to_bits(Y)
    assert gemm_tolerance_failures(Yg, Yr, Y64, mag).size == 0


@pytest.mark.parametrize("M", [1, 7, 16])
def test_adversarial(M, w12lib, oracle):
    W = synth.adversarial_weights(300, 1400, seed=40 + M)
    A = synth.activations(M, 1400, seed=41)
    check_parity(oracle, w12lib, W, A)


@pytest.mark.parametrize("split", [1, 2, 3, 7, 22])
def test_forced_splits(split, w12lib, oracle):
    W = synth.dense_weights(256, 1408, seed=50)
    A = synth.activations(6, 1408, seed=51)
    check_parity(oracle, w12lib, W, A, opts=w12lib.make_opts(split_k=split))


def test_exact_single_products(w12lib, oracle):
    rng = np.random.default_rng(60)
    W = synth.dense_weights(64, 1, seed=61, zero_frac=0.05, outlier_frac=0.05)
    A = synth.activations(3, 1, seed=62)
    Ap = np.zeros((3, 8), np.uint16)
    Ap[:, :1] = A
    st, ref = oracle.encode(W)
    st, Yr, _, _ = oracle.gemm(A, ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Y = w12lib.w12_gemm(synth.bits_to_tensor(Ap, "cuda")[:, :1], t)
    assert np.array_equal(synth.tensor_to_bits(Y), Yr)


def test_exact_zero_rows_one_hot_and_small_integers(w12lib, oracle):
    K, N = 256, 96
    rng = np.random.default_rng(63)
    W = np.zeros((N, K), np.uint16)
    for n in range(32, 64):  # one-hot power-of-two rows
        W[n, rng.integers(0, K)] = (127 + int(rng.integers(-6, 7))) << 7
    Wi = rng.integers(-8, 9, size=(32, K)).astype(np.float32)  # small-integer rows
    W[64:] = synth.tensor_to_bits(torch.from_numpy(Wi).to(torch.bfloat16))
    for A in (synth.activations(9, K, seed=64),
              synth.tensor_to_bits(torch.from_numpy(rng.integers(-8, 9, size=(9, K)).astype(np.float32))
                                   .to(torch.bfloat16))):
        st, ref = oracle.encode(W)
        st, Yr, _, _ = oracle.gemm(A, ref)
        Yg, _ = run_gpu(w12lib, W, A)
        assert (Yg[:, :32] == 0).all()
        assert np.array_equal(Yg[:, 32:64], Yr[:, 32:64])  # a single exact product each
    assert np.array_equal(Yg[:, 64:], Yr[:, 64:])  # integer sums below 2^24 are exact in FP32


def test_nonfinite_weights(w12lib, oracle):
    W = synth.dense_weights(32, 512, seed=65)
    W[2, 5] = 0x7F80
    W[3, 9] = 0xFFC1
    W[4, 100] = 0xFF80
    A = synth.activations(4, 512, seed=66)
    A[1, 5] = 0
    check_parity(oracle, w12lib, W, A)


def test_deterministic_across_runs_and_grids(w12lib):
    """The escape stress shape (N=5121, K=17400): ten runs with different
    grid caps, bitwise identical."""
    N, K = 5121, 17400
    W = synth.adversarial_weights(N, K, seed=4)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M in (1, 7, 16):
        A = synth.bits_to_tensor(synth.activations(M, K, seed=70 + M), "cuda")
        outs = []
        for cap in (0, 1, 7, sms // 2, sms, 2 * sms, 3, 0, 64, 5 * sms):
            Y = w12lib.w12_gemm(A, t, opts=w12lib.make_opts(max_ctas=cap))
            outs.append(synth.tensor_to_bits(Y))
        for o in outs[1:]:
            assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("N,K", [(77829, 256), (40003, 296), (9001, 2304)])
def test_ranges_across_stripes(N, K, w12lib, oracle):
    """The small-M kernel cuts the (stripe, 256-column group) units into one
    contiguous range per resident warp.  Here ranges hold several whole
    stripes (K = 256: one group per stripe), start and end inside stripes
    (K = 296: two groups, the second ragged), or hold a few groups of one or
    two stripes (K = 2304).  Every output is compared with the oracle at
    M = 1, 5 and 16 (both kernel variants), and the result is bitwise the
    same for several grid caps."""
    W = synth.dense_weights(N, K, seed=N + K)
    st, ref = oracle.encode(W)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    for M in (1, 5, 16):
        A = synth.activations(M, K, seed=M + K)
        st, Yr, Y64, mag = oracle.gemm(A, ref)
        Ad = synth.bits_to_tensor(A, "cuda")
        outs = [synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=w12lib.make_opts(max_ctas=cap)))
                for cap in (0, 5, 200)]
        bad = gemm_tolerance_failures(outs[0], Yr, Y64, mag)
        assert bad.size == 0, (M, bad[:10])
        for o in outs[1:]:
            assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("M", [1, 9])
def test_ranges_across_stripes_with_many_escapes(M, w12lib, oracle):
    """Escape-heavy weights (2% of entries far outside the window, zero and
    denormal rows: groups with more than 32 escapes) on a shape whose
    stripes are cut by range boundaries (2.3 groups per range)."""
    N, K = 40003, 600
    W = synth.adversarial_weights(N, K, seed=96)
    st, ref = oracle.encode(W)
    A = synth.activations(M, K, seed=97)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    outs = [synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=w12lib.make_opts(max_ctas=cap))) for cap in (0, 9)]
    bad = gemm_tolerance_failures(outs[0], Yr, Y64, mag)
    assert bad.size == 0, bad[:10]
    assert np.array_equal(outs[0], outs[1])


def test_workspace_left_clean_and_reusable(w12lib, oracle):
    """Counters return to zero after each call, so one workspace serves a
    sequence of different shapes."""
    ws = w12lib.Workspace("cuda", 1 << 22)
    for N, K, M in ((512, 2048, 1), (96, 640, 16), (512, 2048, 3), (1024, 1024, 8), (160, 4096, 16),
                    (8192, 1024, 1), (64, 2048, 2), (6144, 512, 9)):
        W = synth.dense_weights(N, K, seed=N + K)
        A = synth.activations(M, K, seed=M)
        st, ref = oracle.encode(W)
        st, Yr, Y64, mag = oracle.gemm(A, ref)
        t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
        Y = w12lib.w12_gemm(synth.bits_to_tensor(A, "cuda"), t, workspace=ws)
        assert gemm_tolerance_failures(synth.tensor_to_bits(Y), Yr, Y64, mag).size == 0
        torch.cuda.synchronize()
        counters = ws.buf[256:256 + 4 * (N // 16)]
        assert int(counters.sum()) == 0
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK


@pytest.mark.parametrize("name,N,K", [("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120),
                                      ("down", 5120, 17408)])
def test_full_size_layers_sampled(name, N, K, w12lib, oracle):
    """27B-class layer shapes at full size, in the launch configuration the
    benchmark uses; 48 sampled outputs per M checked against the oracle
    evaluated one element at a time on the sampled rows."""
    seed = 1000 + [s[0] for s in synth.LAYER_SHAPES].index(name)
    Wd = synth.dense_weights_device(N, K, seed=seed)
    t = w12lib.w12_encode(Wd)
    rng = np.random.default_rng(seed)
    for M in (1, 8, 16):
        Ad = synth.activations_device(M, K, seed=seed + 100 + M)
        Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t))
        ns = rng.choice(N, size=48, replace=False)
        ms = rng.integers(0, M, size=48)
        Wh = synth.tensor_to_bits(Wd[torch.from_numpy(ns).cuda()])
        st, ref = oracle.encode(Wh)
        st, y, y64, mag = oracle.gemm_sample(synth.tensor_to_bits(Ad), ref, ms, np.arange(48))
        assert st == oracle.OK
        assert gemm_tolerance_failures(Y[ms, ns], y, y64, mag).size == 0


def test_k_zero_writes_zeros(w12lib):
    t = w12lib.w12_encode(torch.zeros(40, 0, dtype=torch.bfloat16, device="cuda"))
    for M in (3, 40):
        A = torch.zeros(M, 8, dtype=torch.bfloat16, device="cuda")[:, :0]
        Y = torch.full((M, 40), 5.0, dtype=torch.bfloat16, device="cuda")
        w12lib.w12_gemm(A, t, Y=Y)
        assert (Y == 0).all()


@pytest.mark.parametrize("M", [4, 16, 64])
def test_overlap_flag_on_a_dependent_chain(M, w12lib):
    """With W12_GEMM_OVERLAP_PREVIOUS each GEMM may start streaming weights
    before the previous kernel ends, but it reads A only after that kernel
    completed: a chain where each GEMM consumes the previous Y gives the
    same bits as the chain without the flag."""
    dims = (512, 1024, 768, 256)
    ts = [w12lib.w12_encode(synth.dense_weights_device(dims[i + 1], dims[i], seed=90 + i))
          for i in range(len(dims) - 1)]
    A0 = synth.activations_device(M, dims[0], seed=95)
    ws = w12lib.Workspace("cuda", 1 << 24)

    def chain(flags):
        x = A0
        outs = []
        for t in ts:
            x = w12lib.w12_gemm(x, t, workspace=ws, opts=w12lib.make_opts(flags=flags))
            outs.append(x)
        torch.cuda.synchronize()
        return [synth.tensor_to_bits(o) for o in outs]

    plain = chain(0)
    for _ in range(3):
        over = chain(w12lib.W12_GEMM_OVERLAP_PREVIOUS)
        for a, b in zip(plain, over):
            assert np.array_equal(a, b)


def test_binding_rejects_bad_operands(w12lib):
    """The C side trusts lda / ldy and writes M rows of N outputs, so the
    Python binding refuses operands whose shape, stride or device does not
    match before any pointer reaches the library."""
    t = w12lib.w12_encode(synth.dense_weights_device(64, 512, seed=990))
    A = synth.activations_device(4, 512, seed=991)
    ok = torch.empty(4, 64, dtype=torch.bfloat16, device="cuda")
    w12lib.w12_gemm(A, t, ok)
    bad_y = (torch.empty(4, 63, dtype=torch.bfloat16, device="cuda"),       # too few columns
             torch.empty(3, 64, dtype=torch.bfloat16, device="cuda"),       # too few rows
             torch.empty(64, 4, dtype=torch.bfloat16, device="cuda").t(),   # transposed
             torch.empty(4, 64, dtype=torch.float32, device="cuda"))        # wrong dtype
    ws = w12lib.Workspace("cuda", 1 << 20)
    for Y in bad_y:
        with pytest.raises(ValueError):
            w12lib.w12_gemm(A, t, Y)
        with pytest.raises(ValueError):
            w12lib.GemmCall(A, t, Y, ws)
        with pytest.raises(ValueError):
            w12lib.w12_gemm_noalloc(A, t, Y)
    with pytest.raises(ValueError):
        w12lib.w12_gemm(synth.activations_device(4, 256, seed=992), t)  # K does not match
    with pytest.raises(ValueError):
        w12lib.w12_gemm(torch.empty(512, 4, dtype=torch.bfloat16, device="cuda").t(), t)  # column stride
    with pytest.raises(ValueError):
        w12lib.w12_gemm(A.cpu(), t)
