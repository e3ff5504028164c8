"""Seeded random GEMM shapes on both GPU paths against the oracle.

SpecPilot (arXiv 2611.02501), section 4.1: the W12 GEMM decodes records in
registers and splits its reduction in a fixed order.  Each case draws N, K
(ragged: neither a multiple of 16 nor of 256 in general), M in 1..256, the
weight recipe, the path (automatic, or the tensor-core path forced for
M <= 16), a forced split or none, and the nested 8-bit view flag, from a fixed
seed.  Every output must pass the tolerance rule against the oracle's FP64
sum, and a second run must give the same bits.
"""
import numpy as np
import pytest

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def draw(seed):
    rng = np.random.default_rng(10_000 + seed)
    N = int(rng.integers(1, 1400))
    K = int(rng.integers(1, 3000))
    M = int(rng.choice([1, 2, 3, 5, 8, 9, 13, 16, 17, 31, 40, 64, 77, 128, 129, 200, 256]))
    kind = ["dense", "adversarial"][int(rng.integers(0, 2))]
    force_tc = M <= 16 and rng.random() < 0.3
    split = int(rng.choice([0, 0, 0, 1, 2, 3, 7]))
    nested = rng.random() < 0.25
    return N, K, M, kind, force_tc, split, nested


@pytest.mark.parametrize("seed", range(32))
def test_random_gemm_against_oracle(seed, w12lib, oracle):
    N, K, M, kind, force_tc, split, nested = draw(seed)
    Kpad = (K + 7) // 8 * 8  # activation rows must be 16-byte aligned
    W = (synth.dense_weights if kind == "dense" else synth.adversarial_weights)(N, K, seed=seed)
    A = np.zeros((M, Kpad), np.uint16)
    A[:, :K] = synth.activations(M, K, seed=seed + 1)
    st, ref = oracle.encode(W)
    assert st == oracle.OK
    Ac = np.ascontiguousarray(A[:, :K])
    st, Yr, Y64, mag = (oracle.gemm_nested8 if nested else oracle.gemm)(Ac, ref)
    assert st == oracle.OK
    flags = w12lib.W12_GEMM_NESTED8 if nested else 0
    opts = w12lib.make_opts(split_k=split, path=w12lib.W12_PATH_TC if force_tc else w12lib.W12_PATH_AUTO,
                            flags=flags)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")[:, :K]
    Y1 = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=opts))
    Y2 = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=opts))
    bad = gemm_tolerance_failures(Y1, Yr, Y64, mag)
    assert bad.size == 0, ((N, K, M, kind, force_tc, split, nested), bad[:8])
    assert np.array_equal(Y1, Y2)
