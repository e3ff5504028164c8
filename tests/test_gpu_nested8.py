"""GPU GEMM on the nested 8-bit view (W12_GEMM_NESTED8) against the oracle.

SpecPilot (arXiv 2611.02501), section 4.1, and the news article's two-level
verification: the low-precision pass reads the 8-bit weight view nested in
W12, i.e. only the hi plane; every weight w acts as w & 0xFFF0 (escapes
included, by this library's reading).  Parity as for the exact GEMM (2 BF16
ulp of the oracle's rounded FP64 sum, or 1e-3 * sum|a||v|), against the
oracle's nested-view GEMM.  Because the view is the truncated tensor, the
GPU result must also equal, bit for bit, the exact GPU GEMM of a tensor
encoded from W & 0xFFF0 (same kernels, same values, same summation order).
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def nested(w12lib, **kw):
    return w12lib.make_opts(flags=w12lib.W12_GEMM_NESTED8, **kw)


@pytest.mark.parametrize("N,K,M", [(1024, 1024, 1), (333, 600, 5), (130, 257 + 7, 8), (300, 1400, 9),
                                   (512, 2048, 16), (640, 1024, 24), (256, 3072, 64), (384, 512, 128)])
@pytest.mark.parametrize("kind", ["dense", "adversarial"])
def test_nested8_parity(N, K, M, kind, w12lib, oracle):
    W = (synth.dense_weights if kind == "dense" else synth.adversarial_weights)(N, K, seed=N + K + M)
    A = synth.activations(M, K, seed=M + 7)
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm_nested8(A, ref)
    assert st == oracle.OK
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=nested(w12lib)))
    bad = gemm_tolerance_failures(Y, Yr, Y64, mag)
    assert bad.size == 0, (bad[:10], Y.reshape(-1)[bad[:10]], Yr.reshape(-1)[bad[:10]])
    # the view is the truncated tensor: the exact GEMM of W & 0xFFF0 gives the same bits
    tt = w12lib.w12_encode(synth.bits_to_tensor(W & 0xFFF0, "cuda"))
    Yt = synth.tensor_to_bits(w12lib.w12_gemm(Ad, tt))
    assert np.array_equal(Y, Yt)


def test_nested8_balanced_ranges(w12lib, oracle):
    """Mpad > 128 on 2432 (row tile, group) units: the balanced-range kernel."""
    W = synth.adversarial_weights(9728, 8192, seed=146)
    A = synth.activations(136, 8192, seed=147)
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm_nested8(A, ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Y = synth.tensor_to_bits(w12lib.w12_gemm(synth.bits_to_tensor(A, "cuda"), t, opts=nested(w12lib)))
    assert gemm_tolerance_failures(Y, Yr, Y64, mag).size == 0


def test_nested8_two_ctas_per_sm(w12lib, oracle):
    """A split-9 grid of 288 CTAs: the tensor-core build with two CTAs per SM."""
    W = synth.adversarial_weights(4096, 2304, seed=144)
    A = synth.activations(40, 2304, seed=145)
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm_nested8(A, ref)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=nested(w12lib, split_k=9)))
    assert gemm_tolerance_failures(Y, Yr, Y64, mag).size == 0
    tt = w12lib.w12_encode(synth.bits_to_tensor(W & 0xFFF0, "cuda"))
    assert np.array_equal(Y, synth.tensor_to_bits(w12lib.w12_gemm(Ad, tt, opts=w12lib.make_opts(split_k=9))))


@pytest.mark.parametrize("M", [1, 16, 48])
def test_nested8_deterministic_across_grids(M, w12lib):
    N, K = 5121, 4000
    t = w12lib.w12_encode(synth.bits_to_tensor(synth.adversarial_weights(N, K, seed=140), "cuda"))
    A = synth.activations_device(M, K, seed=141)
    outs = [synth.tensor_to_bits(w12lib.w12_gemm(A, t, opts=nested(w12lib, max_ctas=cap)))
            for cap in (0, 3, 77, 500)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_nested8_differs_from_exact_only_through_the_low_nibbles(w12lib):
    """Weights whose low mantissa nibbles are already zero: both passes agree."""
    W = synth.dense_weights(2048, 2048, seed=142) & 0xFFF0
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    for M in (3, 40):
        A = synth.activations_device(M, 2048, seed=143 + M)
        a = synth.tensor_to_bits(w12lib.w12_gemm(A, t))
        b = synth.tensor_to_bits(w12lib.w12_gemm(A, t, opts=nested(w12lib)))
        assert np.array_equal(a, b)
