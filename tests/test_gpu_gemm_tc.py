"""GPU W12 GEMM on the tcgen05/TMEM path (M up to 256) against the oracle.

SpecPilot (arXiv 2611.02501), section 4.1: the verify GEMM of tree / block
verification runs with many rows; this path decodes W12 tiles into shared
memory for tcgen05.mma.  Same parity rule as the small-M path
(tests/w12_tol.py) and bitwise determinism across runs.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def parity(w12lib, oracle, W, A, opts=None, reps=1):
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    assert st == oracle.OK
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    outs = []
    for _ in range(reps):
        outs.append(synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=opts)))
    bad = gemm_tolerance_failures(outs[0], Yr, Y64, mag)
    assert bad.size == 0, (bad[:10], outs[0].reshape(-1)[bad[:10]], Yr.reshape(-1)[bad[:10]])
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    return outs[0]


# M > 128 spans the one-CTA build's ring depths (Mpad 144: 5 activation stages, 176-192: 4,
# 208-256: 3; four decoded-A stages)
@pytest.mark.parametrize("M", [17, 24, 32, 33, 48, 63, 64, 128, 136, 168, 184, 200, 232, 256])
def test_tc_dense_1024(M, w12lib, oracle):
    W = synth.dense_weights(1024, 1024, seed=0)
    A = synth.activations(M, 1024, seed=3000 + M)
    parity(w12lib, oracle, W, A, reps=2)


@pytest.mark.parametrize("M", [1, 5, 8, 16])
def test_tc_forced_small_m(M, w12lib, oracle):
    W = synth.dense_weights(512, 2048, seed=1)
    A = synth.activations(M, 2048, seed=3100 + M)
    parity(w12lib, oracle, W, A, opts=w12lib.make_opts(path=w12lib.W12_PATH_TC))


@pytest.mark.parametrize("N,K,M", [(300, 1000, 40), (129, 64, 17), (1, 1, 20), (200, 17400, 33), (77, 260, 256)])
def test_tc_ragged(N, K, M, w12lib, oracle):
    Kpad = (K + 7) // 8 * 8
    W = synth.dense_weights(N, K, seed=N + K)
    A = np.zeros((M, Kpad), np.uint16)
    A[:, :K] = synth.activations(M, K, seed=K + M)
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(np.ascontiguousarray(A[:, :K]), ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Y = w12lib.w12_gemm(synth.bits_to_tensor(A, "cuda")[:, :K], t)
    assert gemm_tolerance_failures(synth.tensor_to_bits(Y), Yr, Y64, mag).size == 0


@pytest.mark.parametrize("split", [1, 2, 5, 8])
def test_tc_forced_splits(split, w12lib, oracle):
    W = synth.dense_weights(384, 2048, seed=2)
    A = synth.activations(40, 2048, seed=3200)
    parity(w12lib, oracle, W, A, opts=w12lib.make_opts(split_k=split), reps=2)


# Grids of at least 258 CTAs with Mpad <= 128 run two CTAs per SM (8 decoder
# warps each, one per stripe, every k-block); smaller grids one CTA per SM
# with 16.  N = 4096 has 32 row tiles: a forced split of 9 gives 288 CTAs,
# one of 8 gives 256.
@pytest.mark.parametrize("M,split", [(40, 9), (40, 8), (17, 9), (128, 9), (129, 9)])
@pytest.mark.parametrize("kind", ["dense", "adversarial"])
def test_tc_both_builds(M, split, kind, w12lib, oracle):
    N, K = 4000, 2304 + 40  # ragged rows and columns; 10 column groups
    W = (synth.dense_weights if kind == "dense" else synth.adversarial_weights)(N, K, seed=M + split)
    A = synth.activations(M, K, seed=3400 + M)
    parity(w12lib, oracle, W, A, opts=w12lib.make_opts(split_k=split), reps=2)


# Balanced ranges (Mpad > 128 and >= 16 units of (128-row tile, 256-column
# group) per SM): 152 contiguous ranges of units, one per CTA.  A range's
# first and last pieces are partial (summed in range order by the row
# tile's last arriving CTA); the row tiles in between are stored directly.
@pytest.mark.parametrize("N,K,M,kind", [
    (9728, 8192, 136, "dense"),         # 76 x 32 = 2432 units, 16 per range: 2 pieces per range
    (9700, 8192, 256, "adversarial"),   # ragged last row tile
    (31232, 2560, 144, "dense"),        # 244 x 10 units, ranges of ~1.6 row tiles
    (9728, 8000, 160, "adversarial"),   # ragged K (Kp = 8192): zero-padded columns in the last group
])
def test_tc_balanced_ranges(N, K, M, kind, w12lib, oracle):
    W = (synth.dense_weights if kind == "dense" else synth.adversarial_weights)(N, K, seed=N + M)
    A = synth.activations(M, K, seed=3600 + M)
    parity(w12lib, oracle, W, A, reps=2)


@pytest.mark.parametrize("M", [200, 256])
def test_tc_automatic_split_above_128(M, w12lib, oracle):
    """8 row tiles, K = 8192: above Mpad = 128 the automatic split is capped at 0.15*K/Mpad
    (5 chunks at M = 200, 4 at M = 256), summed in chunk order."""
    W = synth.dense_weights(1024, 8192, seed=7)
    A = synth.activations(M, 8192, seed=3700 + M)
    parity(w12lib, oracle, W, A, reps=2)


def test_tc_two_per_sm_automatic_split(w12lib, oracle):
    """QKV-sized layer at M = 24: the automatic split (5) fills two CTAs per SM."""
    W = synth.dense_weights(7168, 5120, seed=1000)
    A = synth.activations(24, 5120, seed=3500)
    parity(w12lib, oracle, W, A, reps=2)


def test_tc_adversarial_m33(w12lib, oracle):
    W = synth.adversarial_weights(400, 1496, seed=33)
    A = synth.activations(33, 1496, seed=3300)
    parity(w12lib, oracle, W, A, reps=3)


def test_tc_nonfinite_weights(w12lib, oracle):
    W = synth.dense_weights(130, 512, seed=65)
    W[2, 5] = 0x7F80
    W[3, 9] = 0xFFC1
    W[129, 100] = 0xFF80
    A = synth.activations(20, 512, seed=66)
    A[1, 5] = 0
    parity(w12lib, oracle, W, A)


def test_tc_workspace_error_word_clear(w12lib, oracle):
    ws = w12lib.Workspace("cuda", 1 << 24)
    W = synth.dense_weights(1024, 2048, seed=3)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    for M in (24, 64, 130):
        A = synth.bits_to_tensor(synth.activations(M, 2048, seed=M), "cuda")
        w12lib.w12_gemm(A, t, workspace=ws)
    torch.cuda.synchronize()
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK
    assert int(ws.buf[256:256 + 4 * 64].sum()) == 0


@pytest.mark.parametrize("name,N,K", [("o", 5120, 5120), ("down", 5120, 17408), ("gate_up", 34816, 5120)])
def test_tc_full_size_layers_sampled(name, N, K, w12lib, oracle):
    seed = 1000 + [s[0] for s in synth.LAYER_SHAPES].index(name)
    Wd = synth.dense_weights_device(N, K, seed=seed)
    t = w12lib.w12_encode(Wd)
    rng = np.random.default_rng(seed)
    for M in (24, 64, 256):
        Ad = synth.activations_device(M, K, seed=seed + 200 + M)
        Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t))
        ns = rng.choice(N, size=32, replace=False)
        ms = rng.integers(0, M, size=32)
        Wh = synth.tensor_to_bits(Wd[torch.from_numpy(ns).cuda()])
        st, ref = oracle.encode(Wh)
        st, y, y64, mag = oracle.gemm_sample(synth.tensor_to_bits(Ad), ref, ms, np.arange(32))
        assert gemm_tolerance_failures(Y[ms, ns], y, y64, mag).size == 0
