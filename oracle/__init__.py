"""W12 oracle: plain CPU reference for the W12 format and GEMM.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark may import this package.  The product path
(the CUDA library and its Python binding) never imports or calls it.

The arithmetic lives in ``w12_oracle.c`` (plain C, OpenMP over rows, results
independent of the thread count).  This module compiles it with gcc on first
use and wraps it with ctypes over numpy arrays.

Every function follows "SpecPilot" (arXiv 2611.02501), section 4.1 (W12):
sign bit + 4-bit exponent offset inside a 16-binade window per output
channel + 7 mantissa bits, an exact escape list for out-of-window weights,
zeros and denormals, bit-exact decode, and a GEMM whose exact result is the
FP64 sum of the BF16 products rounded once to BF16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w12_oracle.c")
_LIB = os.path.join(_HERE, "libw12oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID, ERR_CAPACITY, ERR_MISMATCH, ERR_CORRUPT = 0, -1, -3, -5, -7


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc -O2, OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        sig = {
            "w12ref_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "w12ref_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "w12ref_rows_padded": (i64, [i64]),
            "w12ref_cols_padded": (i64, [i64]),
            "w12ref_hi_bytes": (i64, [i64, i64]),
            "w12ref_lo_bytes": (i64, [i64, i64]),
            "w12ref_hi_offset": (i64, [i64, i64, i64]),
            "w12ref_lo_position": (None, [i64, i64, i64, p, p]),
            "w12ref_window_base": (ctypes.c_int, [p, i64]),
            "w12ref_is_escape": (ctypes.c_int, [ctypes.c_uint16, ctypes.c_int]),
            "w12ref_record": (ctypes.c_int, [ctypes.c_uint16, ctypes.c_int]),
            "w12ref_decode_record": (ctypes.c_uint16, [ctypes.c_int, ctypes.c_int]),
            "w12ref_groups": (i64, [i64]),
            "w12ref_ptr_len": (i64, [i64, i64]),
            "w12ref_key": (ctypes.c_int, [i64, i64]),
            "w12ref_encode": (ctypes.c_int, [p, i64, i64, i64, p, p, p, p, p, i64, p]),
            "w12ref_check_structure": (i64, [i64, i64, p, p, i64, i64]),
            "w12ref_decode": (ctypes.c_int, [i64, i64, p, p, p, p, p, i64, p, i64]),
            "w12ref_verify": (ctypes.c_int, [p, i64, i64, i64, p, p, p, p, p, i64, i64, p]),
            "w12ref_gemm": (ctypes.c_int, [p, i64, i64, i64, i64, p, p, p, p, p, i64, p, i64, p, p]),
            "w12ref_gemm_sample": (ctypes.c_int, [p, i64, i64, i64, i64, p, p, p, p, p, i64,
                                                  p, p, i64, p, p, p]),
            "w12ref_decode_nested8": (ctypes.c_int, [i64, i64, p, p, p, p, i64, p, i64]),
            "w12ref_gemm_nested8": (ctypes.c_int, [p, i64, i64, i64, i64, p, p, p, p, i64, p, i64, p, p]),
            "w12ref_gemm_silu_mul": (ctypes.c_int, [p, i64, i64, i64, i64, p, p, p, p, p, i64, p, i64,
                                                    p, p, p, p]),
            "w12ref_round_bf16": (None, [p, i64, p]),
            "w12ref_bits_per_weight": (ctypes.c_double, [i64, i64, i64]),
            "w12ref_num_threads": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return ctypes.c_void_p(a.ctypes.data)


@dataclass
class W12Ref:
    """A W12 tensor held in host memory (numpy arrays)."""
    N: int
    K: int
    hi: np.ndarray        # uint8 [Np*Kp]
    lo: np.ndarray        # uint8 [Np*Kp/2]
    base: np.ndarray      # uint8 [N]
    esc_ptr: np.ndarray   # int32 [Np/16 * groups(K) + 1]
    esc: np.ndarray       # uint32 [esc_cap]: key << 16 | raw BF16 bits
    n_esc: int

    @property
    def esc_key(self) -> np.ndarray:
        return (self.esc >> 16).astype(np.uint16)

    @property
    def esc_val(self) -> np.ndarray:
        return (self.esc & 0xFFFF).astype(np.uint16)

    def bits_per_weight(self) -> float:
        return bits_per_weight(self.N, self.K, self.n_esc)

    def copy(self) -> "W12Ref":
        return W12Ref(self.N, self.K, self.hi.copy(), self.lo.copy(), self.base.copy(),
                      self.esc_ptr.copy(), self.esc.copy(), self.n_esc)

    def position(self, e: int):
        """(n, k) of escape entry e."""
        G = groups(self.K)
        i = int(np.searchsorted(self.esc_ptr, e, side="right")) - 1
        t, g = divmod(i, G)
        key = int(self.esc[e] >> 16)
        return 16 * t + ((key >> 6) & 15), 256 * g + 64 * (key >> 10) + (key & 63)


def num_threads() -> int:
    return _load().w12ref_num_threads()


def groups(K: int) -> int:
    return _load().w12ref_groups(K)


def ptr_len(N: int, K: int) -> int:
    return _load().w12ref_ptr_len(N, K)


def key(n: int, k: int) -> int:
    return _load().w12ref_key(n, k)


def rows_padded(N: int) -> int:
    return _load().w12ref_rows_padded(N)


def cols_padded(K: int) -> int:
    return _load().w12ref_cols_padded(K)


def hi_offset(n: int, k: int, Kp: int) -> int:
    return _load().w12ref_hi_offset(n, k, Kp)


def lo_position(n: int, k: int, Kp: int):
    b = ctypes.c_int64()
    s = ctypes.c_int()
    _load().w12ref_lo_position(n, k, Kp, ctypes.byref(b), ctypes.byref(s))
    return b.value, s.value


def bf16_to_double(b: int) -> float:
    return _load().w12ref_bf16_to_double(b)


def bf16_from_double(x: float) -> int:
    return _load().w12ref_bf16_from_double(x)


def window_base(row: np.ndarray) -> int:
    row = np.ascontiguousarray(row, dtype=np.uint16)
    return _load().w12ref_window_base(_ptr(row), row.size)


def is_escape(w: int, base: int) -> bool:
    return bool(_load().w12ref_is_escape(w, base))


def record(w: int, base: int) -> int:
    return _load().w12ref_record(w, base)


def decode_record(r: int, base: int) -> int:
    return _load().w12ref_decode_record(r, base)


def bits_per_weight(N: int, K: int, n_esc: int) -> float:
    return _load().w12ref_bits_per_weight(N, K, n_esc)


def encode(W: np.ndarray, esc_cap: int | None = None):
    """Encode BF16 bits W [N,K] (uint16).  Returns (status, W12Ref).  With
    esc_cap=None the escape arrays are sized exactly (one counting pass)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    N, K = W.shape
    lib = _load()
    if esc_cap is None:
        st, t = encode(W, esc_cap=0)
        if st == OK:
            return st, t
        esc_cap = t.n_esc
    hi = np.zeros(lib.w12ref_hi_bytes(N, K), np.uint8)
    lo = np.zeros(lib.w12ref_lo_bytes(N, K), np.uint8)
    base = np.zeros(N, np.uint8)
    esc_ptr = np.zeros(lib.w12ref_ptr_len(N, K), np.int32)
    esc = np.zeros(max(esc_cap, 1), np.uint32)
    n_esc = ctypes.c_int64()
    st = lib.w12ref_encode(_ptr(W), N, K, K, _ptr(hi), _ptr(lo), _ptr(base), _ptr(esc_ptr),
                           _ptr(esc), esc_cap, ctypes.byref(n_esc))
    t = W12Ref(N, K, hi, lo, base, esc_ptr, esc[:esc_cap].copy(), n_esc.value)
    if st == OK:
        t.esc = t.esc[:t.n_esc].copy()
    return st, t


def _tensor_args(t: W12Ref):
    esc = t.esc if t.esc.size else np.zeros(1, np.uint32)
    return (_ptr(t.hi), _ptr(t.lo), _ptr(t.base), _ptr(t.esc_ptr), _ptr(esc))


def check_structure(t: W12Ref) -> int:
    esc = t.esc if t.esc.size else np.zeros(1, np.uint32)
    return _load().w12ref_check_structure(t.N, t.K, _ptr(t.esc_ptr), _ptr(esc), t.n_esc, t.esc.size)


def decode(t: W12Ref):
    """Decode to BF16 bits [N,K].  Returns (status, array)."""
    out = np.zeros((t.N, t.K), np.uint16)
    st = _load().w12ref_decode(t.N, t.K, *_tensor_args(t), t.n_esc, _ptr(out), t.K)
    return st, out


def verify(W: np.ndarray, t: W12Ref):
    """Bitwise load-time check.  Returns (status, n_mismatch)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    nm = ctypes.c_int64()
    st = _load().w12ref_verify(_ptr(W), t.K, t.N, t.K, *_tensor_args(t), t.n_esc,
                               t.esc.size, ctypes.byref(nm))
    return st, nm.value


def gemm(A: np.ndarray, t: W12Ref):
    """Y = A * W^T.  Returns (status, Y bf16 bits [M,N], Y64 [M,N], absdot [M,N])."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    M = A.shape[0]
    Y = np.zeros((M, t.N), np.uint16)
    Y64 = np.zeros((M, t.N), np.float64)
    mag = np.zeros((M, t.N), np.float64)
    st = _load().w12ref_gemm(_ptr(A), M, t.K, t.N, t.K, *_tensor_args(t), t.n_esc, _ptr(Y), t.N,
                             _ptr(Y64), _ptr(mag))
    return st, Y, Y64, mag


def gemm_silu_mul(A: np.ndarray, t: W12Ref):
    """The gate/up GEMM with its fused epilogue (reading R24): rows 16s+i
    (gate) and 16s+8+i (up) of W give hidden unit 8s+i; Y[m, 8s+i] =
    BF16(silu(g) * u) from the exact FP64 sums g, u, silu(x) = x/(1+exp(-x))
    in FP64.  Returns (status, Y bits [M, N/2], g64, u64, magG, magU)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    M = A.shape[0]
    H = t.N // 2
    Y = np.zeros((M, H), np.uint16)
    out = [np.zeros((M, H), np.float64) for _ in range(4)]
    st = _load().w12ref_gemm_silu_mul(_ptr(A), M, t.K, t.N, t.K, *_tensor_args(t), t.n_esc, _ptr(Y), H,
                                      *(_ptr(o) for o in out))
    return (st, Y, *out)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Doubles rounded to BF16 bits (nearest, ties to even), element-wise."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, np.uint16)
    _load().w12ref_round_bf16(_ptr(x), x.size, _ptr(out))
    return out


def _nested8_args(t: W12Ref):
    esc = t.esc if t.esc.size else np.zeros(1, np.uint32)
    return _ptr(t.hi), _ptr(t.base), _ptr(t.esc_ptr), _ptr(esc)


def decode_nested8(t: W12Ref):
    """The nested 8-bit view as BF16 bits [N,K] (hi plane + base; escapes
    truncated to 3 mantissa bits).  Returns (status, array)."""
    out = np.zeros((t.N, t.K), np.uint16)
    st = _load().w12ref_decode_nested8(t.N, t.K, *_nested8_args(t), t.n_esc, _ptr(out), t.K)
    return st, out


def gemm_nested8(A: np.ndarray, t: W12Ref):
    """Y = A * V^T with V the nested 8-bit view.  Returns (status, Y, Y64, absdot)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    M = A.shape[0]
    Y = np.zeros((M, t.N), np.uint16)
    Y64 = np.zeros((M, t.N), np.float64)
    mag = np.zeros((M, t.N), np.float64)
    st = _load().w12ref_gemm_nested8(_ptr(A), M, t.K, t.N, t.K, *_nested8_args(t), t.n_esc, _ptr(Y), t.N,
                                     _ptr(Y64), _ptr(mag))
    return st, Y, Y64, mag


def gemm_sample(A: np.ndarray, t: W12Ref, ms, ns):
    """The GEMM at the listed positions only.  Returns (status, y, y64, absdot)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.zeros(ms.size, np.uint16)
    y64 = np.zeros(ms.size, np.float64)
    mag = np.zeros(ms.size, np.float64)
    st = _load().w12ref_gemm_sample(_ptr(A), A.shape[0], A.shape[1], t.N, t.K, *_tensor_args(t),
                                    t.n_esc, _ptr(ms), _ptr(ns), ms.size, _ptr(y), _ptr(y64),
                                    _ptr(mag))
    return st, y, y64, mag
