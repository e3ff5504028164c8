"""Pins for the oracle's nested 8-bit view and its GEMM (CPU only).

SpecPilot (arXiv 2611.02501), section 4.1, and the news article's
"two-level verification": a low-precision pass reads the 8-bit weight view
nested in W12.  The hi byte of a record is sign | 4-bit offset | top 3
mantissa bits, so for an in-window weight the view is
(-1)^s * 2^(base+off-127) * (1 + m_hi/8).  At escaped positions the pages are
silent; the reading taken is the escape's BF16 bits with the 4 low mantissa
bits cleared.  Together: the view of every weight w is w & 0xFFF0.  These
tests pin the hi-plane decode to that closed form on every BF16 pattern, and
the view's GEMM to the exact GEMM of an independently encoded truncated
tensor.
"""
import numpy as np

from lossless_bit_weight_02_gb300 import synth


def test_view_is_truncation_on_every_pattern(oracle):
    """Every BF16 bit pattern (as escapes, and in windows of many bases)."""
    W = synth.all_patterns(64, seed=11)
    st, t = oracle.encode(W)
    st, V = oracle.decode_nested8(t)
    assert st == oracle.OK
    assert np.array_equal(V, W & 0xFFF0)
    # rows whose weights all sit in one window: every base from 1 to 239
    rng = np.random.default_rng(12)
    rows = []
    for base in range(1, 240):
        e = base + rng.integers(0, 16, size=256)
        rows.append((rng.integers(0, 2, size=256) << 15) | (e << 7) | rng.integers(0, 128, size=256))
    W2 = np.array(rows, dtype=np.uint16)
    st, t2 = oracle.encode(W2)
    assert t2.n_esc == 0
    st, V2 = oracle.decode_nested8(t2)
    assert np.array_equal(V2, W2 & 0xFFF0)


def test_view_closed_form(oracle):
    """(-1)^s * 2^(base+off-127) * (1 + m_hi/8) from the record fields."""
    W = synth.dense_weights(40, 500, seed=13, zero_frac=0, outlier_frac=0)
    st, t = oracle.encode(W)
    st, V = oracle.decode_nested8(t)
    Wd = oracle.decode(t)[1]
    assert np.array_equal(Wd, W)
    for n in range(0, 40, 7):
        base = int(t.base[n])
        for k in range(0, 500, 37):
            w = int(W[n, k])
            if oracle.is_escape(w, base):
                continue
            r = oracle.record(w, base)
            s, off, mh = r >> 11, (r >> 7) & 15, (r & 127) >> 4
            want = (-1.0) ** s * 2.0 ** (base + off - 127) * (1.0 + mh / 8.0)
            assert oracle.bf16_to_double(int(V[n, k])) == want


def test_view_gemm_equals_exact_gemm_of_truncated_tensor(oracle):
    for N, K, M, seed in ((96, 448, 5, 14), (33, 1000, 3, 15), (64, 256, 16, 16)):
        W = synth.adversarial_weights(N, K, seed=seed)
        A = synth.activations(M, K, seed=seed + 100)
        st, t = oracle.encode(W)
        st, Yq, Yq64, magq = oracle.gemm_nested8(A, t)
        assert st == oracle.OK
        st, tt = oracle.encode(W & 0xFFF0)
        st, Y, Y64, mag = oracle.gemm(A, tt)
        assert np.array_equal(Yq, Y)
        assert np.array_equal(Yq64, Y64, equal_nan=True)
        assert np.array_equal(magq, mag, equal_nan=True)


def test_view_gemm_is_exact_gemm_when_low_nibbles_are_zero(oracle):
    W = synth.dense_weights(48, 320, seed=17) & 0xFFF0
    A = synth.activations(4, 320, seed=18)
    st, t = oracle.encode(W)
    assert np.array_equal(oracle.gemm_nested8(A, t)[1], oracle.gemm(A, t)[1])
