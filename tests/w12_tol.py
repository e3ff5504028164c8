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


def silu_mul_tolerance_failures(y_bits, ref_bits, g64, u64, mag_g, mag_u):
    """Rule for the fused gate/up epilogue y = silu(g) * u (reading R24).

    The GPU forms g and u as FP32 sums: by the GEMM rule each lies within
    e_g = 1e-3 * sum|a||w_g| (e_u likewise) of the FP64 sums g64, u64.  With
    |silu'| <= 1.1, silu(g) * u then moves by at most
        (|silu(g64)| + 1.1 e_g) e_u + 1.1 e_g |u64|,
    the FP32 evaluation adds a few FP32 ulps (1e-6 relative) and the final
    rounding half a BF16 ulp.  An element passes if it is within that bound
    (plus one BF16 ulp) of the FP64 value, or within 2 BF16 ulp of the
    oracle's BF16 result.  Non-finite references must match in class."""
    y = bf16_bits_to_f64(np.asarray(y_bits)).reshape(-1)
    r = bf16_bits_to_f64(np.asarray(ref_bits)).reshape(-1)
    g = np.asarray(g64, np.float64).reshape(-1)
    u = np.asarray(u64, np.float64).reshape(-1)
    eg = 1e-3 * np.asarray(mag_g, np.float64).reshape(-1)
    eu = 1e-3 * np.asarray(mag_u, np.float64).reshape(-1)
    with np.errstate(over="ignore", invalid="ignore"):
        s = g / (1.0 + np.exp(-g))
        y64 = s * u
        bound = (np.abs(s) + 1.1 * eg) * eu + 1.1 * eg * np.abs(u) + 1e-6 * np.abs(y64) + ulp_bf16(y64)
        ok_num = np.isfinite(y) & ((np.abs(y - r) <= 2 * ulp_bf16(r)) | (np.abs(y - y64) <= bound))
    fin = np.isfinite(y64)
    same_class = (np.isnan(r) & np.isnan(y)) | (np.isinf(r) & np.isinf(y) & (np.sign(r) == np.sign(y)))
    ok = np.where(fin, ok_num, same_class)
    return np.nonzero(~ok)[0]
