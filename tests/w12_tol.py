"""GEMM tolerance rule and small helpers shared by the GPU tests.

Rule (for every output element): pass if
    |y - y_ref_bf16| <= 2 * ulp_bf16(y_ref_bf16)        (ulp of 0 = ulp at 2^-126)
 or |y - y_ref64|    <= 1e-3 * sum_k |a_k| |w_k|
where y_ref_bf16 is the oracle's FP64 sum rounded once to BF16 and y_ref64
the FP64 sum itself.  Non-finite references must match in class and sign;
elements whose FP64 sum or magnitude sum exceeds the FP32 range are exempt
from the numeric bound (FP32 partial sums may overflow where FP64 does not).
"""
import numpy as np
import torch

FLT_MAX = float(np.finfo(np.float32).max)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """BF16 ulp of each value (non-finite values get an infinite ulp)."""
    a = np.where(np.isfinite(v), np.abs(v), 0.0)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(np.where(a > 0, e, -126.0), -126.0)
    return np.where(np.isfinite(v), np.ldexp(1.0, (e - 7).astype(np.int64)), np.inf)


def gemm_tolerance_failures(y_bits, ref_bits, y64, absdot):
    """Returns the flat indices of elements that break the rule."""
    y = bf16_bits_to_f64(np.asarray(y_bits)).reshape(-1)
    r = bf16_bits_to_f64(np.asarray(ref_bits)).reshape(-1)
    y64 = np.asarray(y64, np.float64).reshape(-1)
    mag = np.asarray(absdot, np.float64).reshape(-1)
    fin64 = np.isfinite(y64)
    with np.errstate(invalid="ignore"):
        exempt = fin64 & ((np.abs(y64) > FLT_MAX) | ~np.isfinite(mag) | (mag > FLT_MAX))
        ok_num = np.isfinite(y) & ((np.abs(y - r) <= 2 * ulp_bf16(r)) | (np.abs(y - y64) <= 1e-3 * mag))
    same_inf = np.isinf(r) & np.isinf(y) & (np.sign(r) == np.sign(y))
    same_nan = np.isnan(r) & np.isnan(y)
    ok_class = same_inf | same_nan
    ok = np.where(fin64, ok_num | same_inf | exempt, ok_class)
    return np.nonzero(~ok)[0]
