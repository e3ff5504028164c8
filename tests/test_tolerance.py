"""The GEMM tolerance rule itself rejects planted mistakes (CPU only)."""
import numpy as np
import torch

from w12_tol import gemm_tolerance_failures, ulp_bf16


def bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_ulp():
    assert ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133
    assert ulp_bf16(np.array([-3.0]))[0] == 2.0 ** -6


def test_rule_accepts_and_rejects():
    ref = np.array([1.0, 1.0, 1.0, 100.0, 0.0, float("inf"), float("nan"), 1.0])
    y64 = np.array([1.0, 1.0, 1.0, 100.0, 0.0, float("inf"), float("nan"), 1.0])
    mag = np.array([1e-6, 1e-6, 5e3, 1e-6, 0.0, float("inf"), float("inf"), 1e-6])
    y = np.array([1.0 + 2 * 2 ** -7, 1.0 + 3 * 2 ** -7, 1.0 + 3 * 2 ** -7, 101.0, 2.0 ** -120,
                  float("inf"), float("nan"), float("nan")])
    bad = gemm_tolerance_failures(bits(y), bits(ref), y64, mag)
    # element 1: 3 ulp with a tiny magnitude sum; 4: 2^-120 for an exact 0;
    # 7: NaN for a finite reference
    assert bad.tolist() == [1, 4, 7]


def test_rule_inf_sign_and_overflow_exemption():
    ref = np.array([float("inf"), 3e38])
    y64 = np.array([float("inf"), 3.3e38])
    mag = np.array([float("inf"), 4e38])  # above FLT_MAX: exempt
    y = np.array([-float("inf"), float("inf")])
    assert gemm_tolerance_failures(bits(y), bits(ref), y64, mag).tolist() == [0]
