"""Pins for the oracle GEMM (CPU only).

The oracle's Y = A * W^T (SpecPilot, arXiv 2611.02501, section 4.1: BF16
activations times W12 weights, FP32-or-better accumulation, BF16 out) is
checked against torch's float64 matmul of the decoded weights, and against
cases whose result is exact and known in closed form.
"""
import numpy as np
import torch

from lossless_bit_weight_02_gb300 import synth


def bits_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def f64(bits):
    return bits_tensor(bits).to(torch.float64)


def round_f32_to_bf16_bits(x32: torch.Tensor) -> np.ndarray:
    """torch's float32 -> BF16 round-to-nearest-even (one rounding when the
    float32 value is exact)."""
    return x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_gemm_matches_float64_matmul(oracle):
    W = synth.dense_weights(96, 448, seed=31)
    A = synth.activations(5, 448, seed=1031)
    st, t = oracle.encode(W)
    st, Y, Y64, mag = oracle.gemm(A, t)
    assert st == oracle.OK
    ref = f64(A) @ f64(W).T  # torch's library matmul of the original weights
    rel = (torch.from_numpy(Y64) - ref).abs() / ref.abs().clamp_min(1e-300)
    assert float(rel.max()) <= 1e-12
    assert np.allclose(mag, (f64(A).abs() @ f64(W).abs().T).numpy(), rtol=1e-12)
    # the BF16 output is the FP64 sum rounded once: within half a BF16 ulp
    y = f64(Y)
    ulp = torch.ldexp(torch.ones_like(ref), torch.floor(torch.log2(ref.abs())).to(torch.int32) - 7)
    assert bool(((y - torch.from_numpy(Y64)).abs() <= ulp / 2).all())


def test_gemm_single_product_exact(oracle):
    """M=1, K=1: y = bf16(a*w); the product of two BF16 values is exact in
    float32, so torch's float32 -> BF16 cast is a single rounding."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        a = synth.activations(1, 1, seed=int(rng.integers(1 << 30)))
        W = synth.dense_weights(1, 1, seed=int(rng.integers(1 << 30)), zero_frac=0, outlier_frac=0)
        st, t = oracle.encode(W)
        st, Y, _, _ = oracle.gemm(a, t)
        want = round_f32_to_bf16_bits(bits_tensor(a).float() * bits_tensor(W).float())
        assert Y[0, 0] == want[0, 0]


def test_gemm_zero_rows_give_positive_zero(oracle):
    W = synth.dense_weights(32, 128, seed=3)
    W[[0, 7, 31], :] = 0
    A = synth.activations(3, 128, seed=4)
    st, t = oracle.encode(W)
    st, Y, _, _ = oracle.gemm(A, t)
    assert (Y[:, [0, 7, 31]] == 0).all()


def test_gemm_one_hot_power_of_two_rows(oracle):
    """Row n of W = 2^p * e_{c(n)}: Y[:,n] = 2^p * A[:,c(n)] exactly."""
    K, N = 192, 48
    rng = np.random.default_rng(8)
    cols = rng.integers(0, K, N)
    pw = rng.integers(-6, 7, N)
    W = np.zeros((N, K), np.uint16)
    for n in range(N):
        W[n, cols[n]] = (127 + pw[n]) << 7
    A = synth.activations(4, K, seed=9)
    st, t = oracle.encode(W)
    st, Y, _, _ = oracle.gemm(A, t)
    want = (f64(A)[:, cols] * torch.from_numpy(2.0 ** pw)).to(torch.float32)
    assert np.array_equal(Y, round_f32_to_bf16_bits(want))


def test_gemm_small_integers_exact(oracle):
    """Integer A and W with |.| <= 8 and K <= 256: the sum is an exact integer
    (|sum| < 2^24), so the result is that integer rounded once to BF16."""
    rng = np.random.default_rng(10)
    for K in (1, 17, 64, 200, 256):
        Ai = rng.integers(-8, 9, size=(3, K))
        Wi = rng.integers(-8, 9, size=(20, K))
        A = round_f32_to_bf16_bits(torch.from_numpy(Ai.astype(np.float32)))
        W = round_f32_to_bf16_bits(torch.from_numpy(Wi.astype(np.float32)))
        st, t = oracle.encode(W)
        st, Y, Y64, _ = oracle.gemm(A, t)
        exact = Ai @ Wi.T
        assert np.array_equal(Y64, exact.astype(np.float64))
        assert np.array_equal(Y, round_f32_to_bf16_bits(torch.from_numpy(exact.astype(np.float32))))


def test_gemm_sample_equals_full(oracle):
    W = synth.adversarial_weights(70, 333, seed=12)
    A = synth.activations(6, 333, seed=13)
    st, t = oracle.encode(W)
    st, Y, Y64, mag = oracle.gemm(A, t)
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, 6, 50), rng.integers(0, 70, 50)
    st, y, y64, m = oracle.gemm_sample(A, t, ms, ns)
    assert st == oracle.OK
    assert np.array_equal(y, Y[ms, ns])
    assert np.array_equal(y64, Y64[ms, ns], equal_nan=True)
    assert np.array_equal(m, mag[ms, ns], equal_nan=True)


def test_gemm_nonfinite_weights_propagate(oracle):
    W = synth.dense_weights(16, 64, seed=1)
    W[2, 5] = 0x7F80   # +Inf
    W[3, 9] = 0xFFC1   # NaN
    A = synth.activations(2, 64, seed=2)
    A[1, 5] = 0        # 0 * Inf = NaN
    st, t = oracle.encode(W)
    st, Y, _, _ = oracle.gemm(A, t)
    a05 = float(f64(A)[0, 5])
    assert Y[0, 2] == (0x7F80 if a05 > 0 else 0xFF80)
    assert (Y[1, 2] & 0x7FFF) > 0x7F80  # NaN
    assert (Y[0, 3] & 0x7FFF) > 0x7F80 and (Y[1, 3] & 0x7FFF) > 0x7F80
