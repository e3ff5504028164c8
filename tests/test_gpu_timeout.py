"""The bounded waits of the tensor-core GEMM, made to run out on purpose.

Every mbarrier wait in the tcgen05 kernel is bounded (about a second).  With
W12_GEMM_TEST_STALL one wait of the MMA warp waits for an event that never
comes: it gives up, the CTA aborts, drains its own copies and MMAs, frees its
TMEM and records the failure in the workspace error word.  The call returns,
w12_gemm_workspace_status reports W12_ERR_TIMEOUT (and clears it), the
workspace counters stay clean, and the next normal call on the same context
gives the right result.  The encoder's waits are made to run out the same
way (w12_encode_test_stall).  Nothing here traps or faults the GPU.
"""
import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


# one K-chunk; a split of the reduction; a split-9 grid of 288 CTAs (two CTAs
# per SM); 152 balanced ranges (Mpad > 128, 2432 units)
@pytest.mark.parametrize("N,K,split,M", [(1024, 1024, 0, 32), (1024, 8192, 0, 32), (4096, 2304, 9, 32),
                                         (9728, 8192, 0, 136)])
def test_stalled_wait_reports_timeout_and_the_context_stays_usable(N, K, split, M, w12lib, oracle):
    W = synth.dense_weights(N, K, seed=150 + K)
    A = synth.activations(M, K, seed=151)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    ws = w12lib.Workspace("cuda", 1 << 25)

    w12lib.w12_gemm(Ad, t, workspace=ws, opts=w12lib.make_opts(flags=w12lib.W12_GEMM_TEST_STALL, split_k=split))
    torch.cuda.synchronize()
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_ERR_TIMEOUT
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK  # read and cleared
    assert int(ws.buf[256:256 + 4 * 256].sum()) == 0  # no arrival counter left behind

    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    Y = synth.tensor_to_bits(w12lib.w12_gemm(Ad, t, workspace=ws, opts=w12lib.make_opts(split_k=split)))
    torch.cuda.synchronize()
    assert gemm_tolerance_failures(Y, Yr, Y64, mag).size == 0
    assert w12lib.w12_gemm_workspace_status(ws) == w12lib.W12_OK


@pytest.mark.parametrize("N,K", [(64, 1000), (2048, 5120)])
def test_encode_stall_reports_timeout_and_the_next_encode_is_exact(N, K, w12lib, oracle):
    """The encoder's bounded waits (the pack kernel's two grid barriers and its
    look-back): with w12_encode_test_stall on, the pack's block 0 skips the
    first barrier, every block's wait runs out and w12_encode reports
    W12_ERR_TIMEOUT.  The next encode on the same context (hook off) gives the
    oracle's bytes."""
    W = synth.adversarial_weights(N, K, seed=51 + N)
    Wd = synth.bits_to_tensor(W, "cuda")
    lib = w12lib.load()
    lib.w12_encode_test_stall(1)
    try:
        with pytest.raises(w12lib.W12Error) as ei:
            w12lib.w12_encode(Wd)
        assert ei.value.status == w12lib.W12_ERR_TIMEOUT
    finally:
        lib.w12_encode_test_stall(0)
    t = w12lib.w12_encode(Wd)
    torch.cuda.synchronize()
    st, ref = oracle.encode(W)
    assert t.n_esc == ref.n_esc
    assert np.array_equal(t.hi.cpu().numpy(), ref.hi) and np.array_equal(t.lo.cpu().numpy(), ref.lo)
    assert np.array_equal(t.base.cpu().numpy(), ref.base)
    assert np.array_equal(t.esc_ptr.cpu().numpy(), ref.esc_ptr)
    assert np.array_equal(t.esc[:t.n_esc].cpu().numpy().view(np.uint32), ref.esc[:ref.n_esc])
