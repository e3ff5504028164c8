"""Pins of the oracle's fused gate/up epilogue (reading R24).

The exact pass streams a gated MLP, whose gate/up GEMM is followed by
silu(g) * u before the down GEMM (silu(x) = x / (1 + exp(-x))).  The pages do
not write this epilogue out, so the reading is the published SiLU with this
library's row layout: in row stripe t of W, row 16t+i is the gate row and row
16t+8+i the up row of hidden unit 8t+i.  The oracle computes g and u as exact
FP64 sums, silu(g) * u in FP64, and rounds once to BF16.

What pins it, besides itself:
  * a hand-worked fixture (tests/golden/worked_silu_mul.txt) on one-hot rows
    whose values were worked out by hand: fixes the formula, which row is the
    gate and which the up, and the hidden-unit numbering across two stripes;
  * closed cases: g = 0 gives 0; g = 64 gives exactly 64 * u; u = 0 gives 0;
  * the identity silu(g) - silu(-g) = g on gate rows w and -w with u = 1;
  * linearity in u: scaling the up row by 2 (an exact power) doubles y;
  * copies of the epilogue with a planted mistake (gate and up swapped,
    sigmoid without the factor g, rows paired 2i / 2i+1, the sign of the
    exponent flipped, the product with u missing) each fail a pin.
"""
import math
import os

import numpy as np
import pytest

from lossless_bit_weight_02_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
ONE = 0x3F80


def fixture():
    acts, rows = None, []
    for ln in open(os.path.join(HERE, "golden", "worked_silu_mul.txt")):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        parts = ln.split()
        if parts[0] == "activations":
            acts = np.array([int(x, 16) for x in parts[1:]], np.uint16)
        else:
            rows.append((int(parts[0]), int(parts[1]), int(parts[2]), int(parts[3], 16)))
    return acts, rows


def one_hot_weights(rows, K):
    """W [16*stripes, K]: gate row 16t+i picks gate_col, up row 16t+8+i picks up_col."""
    H = len(rows)
    W = np.zeros((2 * H, K), np.uint16)
    for h, gc, uc, _ in rows:
        t, i = divmod(h, 8)
        W[16 * t + i, gc] = ONE
        W[16 * t + 8 + i, uc] = ONE
    return W


# ---- the epilogue under test, and copies of it with a planted mistake ----
# Each maps the oracle's FP64 GEMM output [M, N] (exact sums) to the BF16
# result [M, N/2]; `via_oracle` calls the oracle itself.

def _pairs(N):
    j = np.arange(N // 2)
    gate = (j // 8) * 16 + j % 8
    return gate, gate + 8


def planted_swap(oracle, Y64):
    gate, up = _pairs(Y64.shape[1])
    g, u = Y64[:, up], Y64[:, gate]
    return oracle.round_bf16(g / (1.0 + np.exp(-g)) * u)


def planted_sigmoid_only(oracle, Y64):
    gate, up = _pairs(Y64.shape[1])
    g, u = Y64[:, gate], Y64[:, up]
    return oracle.round_bf16(1.0 / (1.0 + np.exp(-g)) * u)


def planted_adjacent_rows(oracle, Y64):
    j = np.arange(Y64.shape[1] // 2)
    g, u = Y64[:, 2 * j], Y64[:, 2 * j + 1]
    return oracle.round_bf16(g / (1.0 + np.exp(-g)) * u)


def planted_exp_sign(oracle, Y64):
    gate, up = _pairs(Y64.shape[1])
    g, u = Y64[:, gate], Y64[:, up]
    with np.errstate(over="ignore"):
        return oracle.round_bf16(g / (1.0 + np.exp(g)) * u)


def planted_no_up(oracle, Y64):
    gate, up = _pairs(Y64.shape[1])
    g = Y64[:, gate]
    return oracle.round_bf16(g / (1.0 + np.exp(-g)))


PLANTED = (planted_swap, planted_sigmoid_only, planted_adjacent_rows, planted_exp_sign, planted_no_up)


def via_oracle(oracle, A, W):
    st, ref = oracle.encode(W)
    assert st == oracle.OK
    st, Y, g64, u64, mg, mu = oracle.gemm_silu_mul(A, ref)
    assert st == oracle.OK
    return Y


def via_planted(fn):
    def run(oracle, A, W):
        st, ref = oracle.encode(W)
        st, _, Y64, _ = oracle.gemm(A, ref)
        return fn(oracle, Y64)
    return run


# ---- pins, each a function (oracle, epilogue) -> bool ----

def pin_fixture(oracle, epi):
    acts, rows = fixture()
    W = one_hot_weights(rows, acts.size)
    Y = epi(oracle, acts[None, :], W)
    want = np.array([r[3] for r in rows], np.uint16)
    return np.array_equal(np.asarray(Y).reshape(-1), want)


def pin_closed_cases(oracle, epi):
    """g = 0 gives 0; g = 64 gives exactly 64 u (1 + e^-64 is 1 in FP64);
    u = 0 gives a zero with the sign of silu(g)."""
    K = 16
    A = np.zeros((1, K), np.uint16)
    A[0, 0] = 0x4280   # 64
    A[0, 1] = 0x3F40   # 0.75
    A[0, 2] = 0xC0A0   # -5
    W = np.zeros((16, K), np.uint16)
    W[0, 3] = ONE; W[8, 1] = ONE      # g = 0 (column 3 holds 0), u = 0.75 -> +0
    W[1, 0] = ONE; W[9, 1] = ONE      # g = 64, u = 0.75 -> 48
    W[2, 2] = ONE; W[10, 3] = ONE     # g = -5, u = 0 -> -0
    W[3, 0] = ONE; W[11, 2] = ONE     # g = 64, u = -5 -> -320
    Y = np.asarray(epi(oracle, A, W)).reshape(-1)     # units 4..7: g = u = 0 -> +0
    want = np.array([0x0000, 0x4240, 0x8000, 0xC3A0, 0, 0, 0, 0], np.uint16)
    return bool(np.array_equal(Y, want))


def pin_odd_identity(oracle, epi):
    """silu(g) - silu(-g) = g, with u = 1: hidden units 2h and 2h+1 get gate
    rows w and -w."""
    K = 64
    A = synth.activations(1, K, seed=77)
    A[0, K - 1] = ONE  # u = 1 from the last column
    W = np.zeros((32, K), np.uint16)
    w = synth.dense_weights(8, K - 1, seed=78)
    for h in range(8):
        t, i = divmod(2 * h, 8)
        W[16 * t + i, :K - 1] = w[h]
        W[16 * t + 8 + i, K - 1] = ONE
        t, i = divmod(2 * h + 1, 8)
        W[16 * t + i, :K - 1] = w[h] ^ 0x8000
        W[16 * t + 8 + i, K - 1] = ONE
    Y = np.asarray(epi(oracle, A, W)).reshape(-1)
    f = bf16_to_f64(Y)
    a = bf16_to_f64(A[0, :K - 1])
    ok = True
    for h in range(8):
        g = float(np.dot(a, bf16_to_f64(w[h])))
        diff = f[2 * h] - f[2 * h + 1]
        tol = ulp(f[2 * h]) + ulp(f[2 * h + 1])
        ok &= abs(diff - g) <= tol
    return bool(ok)


def pin_linear_in_u(oracle, epi):
    """Doubling the up row (an exact power of two) doubles every output."""
    W = synth.dense_weights(32, 128, seed=90)
    A = synth.activations(2, 128, seed=91)
    W2 = W.copy()
    for t in range(2):
        rows = W2[16 * t + 8:16 * t + 16]
        e = (rows >> 7) & 0xFF
        ok_rows = (e > 0) & (e < 254)
        rows[ok_rows] = rows[ok_rows] + (1 << 7)  # exponent + 1: times 2
        W2[16 * t + 8:16 * t + 16] = rows
    y1 = bf16_to_f64(np.asarray(epi(oracle, A, W)))
    y2 = bf16_to_f64(np.asarray(epi(oracle, A, W2)))
    return bool(np.array_equal(2 * y1, y2))


PINS = (pin_fixture, pin_closed_cases, pin_odd_identity, pin_linear_in_u)


def bf16_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def ulp(v):
    a = abs(v)
    e = math.floor(math.log2(a)) if a > 0 else -126
    return 2.0 ** (max(e, -126) - 7)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_epilogue_pins(pin, oracle):
    assert pin(oracle, via_oracle)


@pytest.mark.parametrize("mistake", PLANTED, ids=lambda p: p.__name__)
def test_planted_mistakes_fail_a_pin(mistake, oracle):
    epi = via_planted(mistake)
    assert not all(pin(oracle, epi) for pin in PINS), mistake.__name__


def test_output_shape_and_bad_n(oracle):
    W = synth.dense_weights(48, 256, seed=3)
    A = synth.activations(3, 256, seed=4)
    st, ref = oracle.encode(W)
    st, Y, g, u, mg, mu = oracle.gemm_silu_mul(A, ref)
    assert st == oracle.OK and Y.shape == (3, 24) and g.shape == (3, 24)
    st, ref = oracle.encode(synth.dense_weights(40, 256, seed=3))
    assert oracle.gemm_silu_mul(A, ref)[0] == oracle.ERR_INVALID  # N not a multiple of 16
