"""The fused gate/up tolerance rule itself: it accepts the oracle's own
result and rejects planted mistakes of the size the rule must catch."""
import numpy as np

from lossless_bit_weight_02_gb300 import synth
from w12_tol import silu_mul_tolerance_failures


def test_rule_accepts_the_reference_and_rejects_mistakes(oracle):
    W = synth.dense_weights(64, 512, seed=11)
    A = synth.activations(4, 512, seed=12)
    st, ref = oracle.encode(W)
    st, Y, g, u, mg, mu = oracle.gemm_silu_mul(A, ref)
    assert silu_mul_tolerance_failures(Y, Y, g, u, mg, mu).size == 0
    # a gate/up swap, a missing silu, a sign flip: each caught on most elements
    st, Ys, *_ = oracle.gemm_silu_mul(A, ref)
    sw = oracle.round_bf16(u / (1 + np.exp(-u)) * g)
    assert silu_mul_tolerance_failures(sw, Y, g, u, mg, mu).size > Y.size // 2
    assert silu_mul_tolerance_failures(oracle.round_bf16(g * u), Y, g, u, mg, mu).size > Y.size // 4
    assert silu_mul_tolerance_failures(Y ^ 0x8000, Y, g, u, mg, mu).size > Y.size // 2
    # one BF16 ulp off is accepted
    assert silu_mul_tolerance_failures(Y + 1, Y, g, u, mg, mu).size == 0
