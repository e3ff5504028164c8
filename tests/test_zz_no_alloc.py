"""w12_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Engines that plan all device memory up front, plug-ins living in another
framework's memory pool and latency-critical loops (where cudaMalloc would
synchronise the device) cannot hand w12_gemm a workspace.  w12_gemm_noalloc
uses the library's built-in scratch array instead.  This test calls it
through the C ABI twice in a row, on two shapes that both use the split-K
scratch, and checks each result against the existing entry point w12_gemm
with the tolerance rule the other GEMM tests use (and, since both run the
same kernels with the same split, bit for bit).

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth
from w12_tol import gemm_tolerance_failures

pytestmark = pytest.mark.gpu


def call_noalloc(w12lib, A, t, Y, opts=None):
    """The raw C-ABI call (no Python helper in between)."""
    lib = w12lib.load()
    s = t.struct()
    o = opts if opts is not None else w12lib.make_opts()
    return lib.w12_gemm_noalloc(ctypes.c_void_p(A.data_ptr()), A.stride(0), ctypes.byref(s),
                                ctypes.c_void_p(Y.data_ptr()), Y.stride(0), A.shape[0], ctypes.byref(o),
                                w12lib._stream())


def test_noalloc_matches_w12_gemm_on_two_calls(w12lib, oracle):
    cases = ((5120, 5120, 8, 81), (1024, 3072, 16, 82))  # both split K: the scratch counters are used
    prepared = []
    for N, K, M, seed in cases:
        assert w12lib.w12_gemm_workspace_bytes(M, N, K) > 256
        W = synth.dense_weights(N, K, seed=seed)
        A = synth.activations(M, K, seed=seed + 1)
        t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
        Ad = synth.bits_to_tensor(A, "cuda")
        Y_ref = w12lib.w12_gemm(Ad, t)  # the existing entry point, with its own workspace
        prepared.append((W, A, t, Ad, Y_ref))
    torch.cuda.synchronize()
    # two calls in a row, nothing in between
    outs = []
    for W, A, t, Ad, Y_ref in prepared:
        Y = torch.full_like(Y_ref, float("nan"))
        assert call_noalloc(w12lib, Ad, t, Y) == w12lib.W12_OK
        outs.append(Y)
    torch.cuda.synchronize()
    for (W, A, t, Ad, Y_ref), Y in zip(prepared, outs):
        st, ref = oracle.encode(W)
        st, _, Y64, mag = oracle.gemm(A, ref)
        got, want = synth.tensor_to_bits(Y), synth.tensor_to_bits(Y_ref)
        assert gemm_tolerance_failures(got, want, Y64, mag).size == 0
        assert np.array_equal(got, want)


def test_noalloc_rejects_work_beyond_its_scratch(w12lib):
    N, K, M = 8192, 4096, 16
    opts = w12lib.make_opts(split_k=16)  # 16 x 8192 x 16 FP32 partials: more than the scratch
    assert w12lib.w12_gemm_workspace_bytes(M, N, K, opts) > w12lib.W12_NOALLOC_SCRATCH_BYTES
    t = w12lib.w12_encode(synth.dense_weights_device(N, K, seed=83))
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(w12lib, A, t, Y, opts) == w12lib.W12_ERR_CAPACITY


def test_noalloc_capacity_of_the_automatic_tensor_core_plan(w12lib):
    """Most automatic tensor-core plans (M > 16) need more split-K partials
    than the scratch holds: M = 17 on a 5120 x 5120 layer gets
    W12_ERR_CAPACITY, and the same shape with split_k = 1 runs."""
    N = K = 5120
    t = w12lib.w12_encode(synth.dense_weights_device(N, K, seed=84))
    A = synth.activations_device(17, K, seed=85)
    Y = torch.zeros(17, N, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(w12lib, A, t, Y) == w12lib.W12_ERR_CAPACITY
    one = w12lib.make_opts(split_k=1)
    assert call_noalloc(w12lib, A, t, Y, one) == w12lib.W12_OK
    ref = w12lib.w12_gemm(A, t, opts=one)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))


def test_noalloc_reports_a_timeout(w12lib, oracle):
    """A bounded wait that gives up inside a w12_gemm_noalloc call (made to
    run out on purpose with W12_GEMM_TEST_STALL on the tensor-core path) is
    reported by w12_gemm_noalloc_status, which reads and clears it; the next
    call is correct again."""
    lib = w12lib.load()
    N, K, M = 1024, 2048, 32
    W = synth.dense_weights(N, K, seed=86)
    A = synth.activations(M, K, seed=87)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    Ad = synth.bits_to_tensor(A, "cuda")
    Y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    stall = w12lib.make_opts(split_k=1, flags=w12lib.W12_GEMM_TEST_STALL)
    assert call_noalloc(w12lib, Ad, t, Y, stall) == w12lib.W12_OK  # asynchronous: the launch succeeded
    assert lib.w12_gemm_noalloc_status(w12lib._stream()) == w12lib.W12_ERR_TIMEOUT
    assert lib.w12_gemm_noalloc_status(w12lib._stream()) == w12lib.W12_OK  # read and cleared
    assert call_noalloc(w12lib, Ad, t, Y, w12lib.make_opts(split_k=1)) == w12lib.W12_OK
    assert lib.w12_gemm_noalloc_status(w12lib._stream()) == w12lib.W12_OK
    st, ref = oracle.encode(W)
    st, Yr, Y64, mag = oracle.gemm(A, ref)
    assert gemm_tolerance_failures(synth.tensor_to_bits(Y), Yr, Y64, mag).size == 0
