"""Bitwise determinism across launch configurations on both GEMM paths.

SpecPilot (arXiv 2611.02501), section 4.1: the W12 GEMM splits its reduction
in a fixed order, so its result is deterministic.  Here "fixed" is taken to
cover the launch configuration too: both kernels cut a GEMM into work items
that depend on (M, N, K) only, and each CTA walks items blockIdx.x,
blockIdx.x + gridDim.x, ..., so capping the grid (w12_gemm_opts.max_ctas)
must leave every output bit unchanged.  Each case runs ten grid caps, from
one CTA to more CTAs than items, and checks the first result against the
oracle with the usual tolerance rule.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu

SMS = 152
GRID_CAPS = (0, 1, 3, 7, SMS // 2, SMS, 2 * SMS, 64, 5 * SMS, 2)


def across_caps(w12lib, oracle, W, A, base_opts=None, caps=GRID_CAPS, sample=None):
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    b = base_opts or w12lib.make_opts()
    outs = []
    for cap in caps:
        o = w12lib.make_opts(max_ctas=cap, split_k=b.split_k, path=b.path, flags=b.flags)
        outs.append(synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=o)))
    for cap, y in zip(caps[1:], outs[1:]):
        assert np.array_equal(y, outs[0]), f"grid cap {cap} changed the result"
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    if b.flags & w12lib.W12_GEMM_NESTED8:
        st, Yr, Y64, mag = oracle.gemm_nested8(A, ref)
    assert gemm_tolerance_failures(outs[0], Yr, Y64, mag).size == 0
    return outs[0]


@pytest.mark.parametrize("M", [1, 7, 16])
def test_small_m_path_across_grids(M, w12lib, oracle):
    W = synth.adversarial_weights(1200, 3000, seed=900 + M)  # ragged N and K, 1-5% escapes
    A = synth.activations(M, 3000, seed=910 + M)
    across_caps(w12lib, oracle, W, A)


# K-chunk kernel: one CTA per SM (16 decoder warps) and two per SM (8), with
# and without a split, ragged rows and columns
@pytest.mark.parametrize("M,split", [(33, 0), (40, 5), (40, 9), (128, 3), (24, 1)])
def test_tc_kchunks_across_grids(M, split, w12lib, oracle):
    W = synth.adversarial_weights(4000, 2344, seed=920 + M + split)
    A = synth.activations(M, 2344, seed=930 + M)
    across_caps(w12lib, oracle, W, A, w12lib.make_opts(split_k=split))


def test_tc_nested8_across_grids(w12lib, oracle):
    W = synth.dense_weights(2048, 4096, seed=940)
    A = synth.activations(64, 4096, seed=941)
    across_caps(w12lib, oracle, W, A, w12lib.make_opts(flags=w12lib.W12_GEMM_NESTED8))


# balanced ranges (Mpad > 128, >= 16 units per SM): ranges cut inside row
# tiles, several ranges per CTA when the grid is capped
@pytest.mark.parametrize("N,K,M", [(9728, 8192, 136), (9700, 8000, 256)])
def test_tc_ranges_across_grids(N, K, M, w12lib, oracle):
    W = synth.adversarial_weights(N, K, seed=950 + M)
    A = synth.activations(M, K, seed=960 + M)
    caps = (0, 1, 2, 5, 76, 151, 152, 300, 64, 3)
    across_caps(w12lib, oracle, W, A, caps=caps)


def test_capped_grid_stall_reports_timeout(w12lib, oracle):
    """A CTA that walks several items and aborts in the first one still ends
    (every later item is skipped) and reports the timeout."""
    W = synth.dense_weights(2048, 4096, seed=970)
    A = synth.activations(32, 4096, seed=971)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    ws = w12lib.Workspace("cuda", 1 << 24)
    for split in (1, 4):
        w12lib.w12_gemm(Ad, t, workspace=ws,
                        opts=w12lib.make_opts(max_ctas=3, split_k=split, flags=w12lib.W12_GEMM_TEST_STALL))
        torch.cuda.synchronize()
        assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_ERR_TIMEOUT
        assert int(ws.buf[256:256 + 4 * 64].sum()) == 0
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, workspace=ws, opts=w12lib.make_opts(max_ctas=3)))
    assert gemm_tolerance_failures(Y, Yr, Y64, mag).size == 0
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK


@pytest.mark.parametrize("M,split", [(40, 3), (64, 5), (24, 2)])
def test_tc_silu_split_across_grids(M, split, w12lib):
    """The fused gate/up epilogue with a split: an uncapped grid (one CTA per
    item; the split's partials summed across a thread-block cluster where the
    clusters fit) and capped grids (partials summed in global memory by the
    row tile's last CTA) add the chunks in the same order, so every output
    bit is the same."""
    N, K = 2 * 1536, 2048
    W = synth.dense_weights(N, K, seed=970 + M)
    A = synth.activations(M, K, seed=980 + M)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    outs = []
    for cap in (0, 5, 2, SMS, 3):
        o = w12lib.make_opts(max_ctas=cap, split_k=split, flags=w12lib.W12_GEMM_SILU_MUL)
        outs.append(synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, opts=o)))
    for y in outs[1:]:
        assert np.array_equal(y, outs[0])
