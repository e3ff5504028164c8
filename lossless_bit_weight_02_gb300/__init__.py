"""W12 for GB300: Python binding of the C-ABI library libw12.so.

W12 is the lossless 12-bit BF16 weight format of "SpecPilot" (arXiv
2611.02501), section 4.1.  Every step of encode, decode, verify and GEMM runs
in the library's CUDA kernels; this module only marshals arguments (torch
tensors -> device pointers, the current CUDA stream) and allocates device
memory through torch.  There is no CPU fallback: if the library cannot be
loaded, every call raises.

Entry points (same names as the C ABI in include/w12.h):
    w12_encode(W)                      -> W12Tensor
    w12_decode(t, out=None)            -> torch.bfloat16 [N,K]
    w12_verify_roundtrip(W, t)         -> (status, n_mismatch)
    w12_gemm(A, t, Y=None, ...)        -> torch.bfloat16 [M,N]
    w12_gemm_workspace_bytes(M, N, K)  -> int
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw12.so")

W12_OK = 0
W12_ERR_INVALID = -1
W12_ERR_ALIGN = -2
W12_ERR_CAPACITY = -3
W12_ERR_CUDA = -4
W12_ERR_MISMATCH = -5
W12_ERR_TIMEOUT = -6
W12_ERR_CORRUPT = -7
W12_ERR_UNSUPPORTED = -8

W12_PATH_AUTO, W12_PATH_MMA, W12_PATH_TC = 0, 1, 2
W12_GEMM_OVERLAP_PREVIOUS = 1
W12_GEMM_NESTED8 = 2  # multiply by the nested 8-bit view (hi plane only)
W12_GEMM_SILU_MUL = 4  # fused gate/up epilogue: Y[m, 8s+i] = silu(row 16s+i) * (row 16s+8+i)
W12_GEMM_TEST_STALL = 1 << 30  # tests only: one bounded wait runs out
W12_LIST_MAX = 64  # GEMMs per launch of w12_gemm_list

# Every symbol include/w12.h declares.
EXPORTS = (
    "w12_rows_padded", "w12_cols_padded", "w12_hi_bytes", "w12_lo_bytes", "w12_groups",
    "w12_esc_ptr_len", "w12_encode", "w12_encode_test_stall",
    "w12_decode", "w12_verify_workspace_bytes", "w12_verify_roundtrip",
    "w12_gemm_workspace_bytes", "w12_gemm", "w12_gemm_noalloc", "w12_gemm_noalloc_status",
    "w12_gemm_workspace_status", "w12_gemm_list_workspace_bytes", "w12_gemm_list",
    "w12_tree_workspace_bytes", "w12_tree_select",
    "w12_gdn_workspace_bytes", "w12_gdn_tree", "w12_gdn_status",
    "w12_status_string", "w12_version",
)

# Size of the scratch array built into the library for w12_gemm_noalloc.
W12_NOALLOC_SCRATCH_BYTES = 4 << 20


class W12Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _Tensor(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("hi", ctypes.c_void_p), ("lo", ctypes.c_void_p), ("base", ctypes.c_void_p),
        ("esc_ptr", ctypes.c_void_p), ("esc", ctypes.c_void_p),
        ("esc_cap", ctypes.c_int64), ("n_esc", ctypes.c_int64),
    ]


class GemmItem(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("w", ctypes.POINTER(_Tensor)),
                ("Y", ctypes.c_void_p), ("ldy", ctypes.c_int64), ("M", ctypes.c_int64),
                ("after", ctypes.c_int32), ("flags", ctypes.c_int32)]


class GemmOpts(ctypes.Structure):
    _fields_ = [("max_ctas", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("path", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libw12.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libw12.so not built ({p}); run __graft_entry__.build() or "
                               "python lossless_bit_weight_02_gb300/_build.py")
        lib = ctypes.CDLL(p)
        i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "w12_rows_padded": (i64, [i64]),
            "w12_cols_padded": (i64, [i64]),
            "w12_hi_bytes": (i64, [i64, i64]),
            "w12_lo_bytes": (i64, [i64, i64]),
            "w12_groups": (i64, [i64]),
            "w12_esc_ptr_len": (i64, [i64, i64]),
            "w12_encode": (st, [vp, i64, ctypes.POINTER(_Tensor), vp]),
            "w12_encode_test_stall": (None, [ctypes.c_int]),
            "w12_decode": (st, [ctypes.POINTER(_Tensor), vp, i64, vp]),
            "w12_verify_workspace_bytes": (sz, []),
            "w12_verify_roundtrip": (st, [vp, i64, ctypes.POINTER(_Tensor), ctypes.POINTER(i64), vp, sz, vp]),
            "w12_gemm_workspace_bytes": (sz, [i64, i64, i64, ctypes.POINTER(GemmOpts)]),
            "w12_gemm": (st, [vp, i64, ctypes.POINTER(_Tensor), vp, i64, i64, vp, sz,
                              ctypes.POINTER(GemmOpts), vp]),
            "w12_gemm_noalloc": (st, [vp, i64, ctypes.POINTER(_Tensor), vp, i64, i64,
                                      ctypes.POINTER(GemmOpts), vp]),
            "w12_gemm_noalloc_status": (st, [vp]),
            "w12_gemm_workspace_status": (st, [vp, sz, vp]),
            "w12_gemm_list_workspace_bytes": (sz, [ctypes.POINTER(GemmItem), ctypes.c_int32,
                                                   ctypes.POINTER(GemmOpts)]),
            "w12_gemm_list": (st, [ctypes.POINTER(GemmItem), ctypes.c_int32, vp, sz, ctypes.POINTER(GemmOpts), vp]),
            "w12_tree_workspace_bytes": (sz, [ctypes.c_int32, ctypes.c_int32]),
            "w12_tree_select": (st, [vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "w12_gdn_workspace_bytes": (sz, [i64, i64, i64, ctypes.c_int32]),
            "w12_gdn_tree": (st, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, sz,
                                  ctypes.c_int32, vp]),
            "w12_gdn_status": (st, [vp, sz, vp]),
            "w12_status_string": (ctypes.c_char_p, [st]),
            "w12_version": (ctypes.c_int32, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().w12_status_string(status).decode()
    except Exception:
        return f"status {status}"


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> ctypes.c_void_p:
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:  # the current stream's handle without building a Stream object
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, what: str):
    if status != W12_OK:
        raise W12Error(status, what)


def _need_cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _out_cols(t: "W12Tensor", flags: int) -> int:
    return t.N // 2 if flags & W12_GEMM_SILU_MUL else t.N


def _check_gemm_operands(A: torch.Tensor, t: "W12Tensor", Y: torch.Tensor | None, flags: int = 0):
    """The C side trusts lda / ldy and writes M rows of N outputs, so the
    shapes, strides and devices are checked here, before any pointer is
    passed: A is [M, K] and Y is [M, N] ([M, N/2] with W12_GEMM_SILU_MUL),
    both with unit column stride, on the device that holds the W12 tensor,
    which must be the current device (the library launches on the current
    device)."""
    if flags & W12_GEMM_SILU_MUL and t.N % 16:
        raise ValueError(f"W12_GEMM_SILU_MUL needs N a multiple of 16, got {t.N}")
    _need_cuda(A, "A", torch.bfloat16)
    if A.dim() != 2 or A.shape[1] != t.K or (A.shape[0] > 0 and t.K > 0 and A.stride(1) != 1):
        raise ValueError(f"A must be [M, {t.K}] with unit column stride, got {tuple(A.shape)} "
                         f"strides {A.stride()}")
    dev = t.hi.device
    if A.device != dev:
        raise ValueError(f"A is on {A.device}, the W12 tensor on {dev}")
    if dev.index != torch.cuda.current_device():
        raise ValueError(f"the W12 tensor is on {dev} but the current device is cuda:{torch.cuda.current_device()}")
    if Y is not None:
        _need_cuda(Y, "Y", torch.bfloat16)
        cols = _out_cols(t, flags)
        if Y.dim() != 2 or tuple(Y.shape) != (A.shape[0], cols) or (Y.numel() > 0 and Y.stride(1) != 1):
            raise ValueError(f"Y must be [{A.shape[0]}, {cols}] with unit column stride, got {tuple(Y.shape)} "
                             f"strides {Y.stride()}")
        if Y.device != dev:
            raise ValueError(f"Y is on {Y.device}, the W12 tensor on {dev}")


@dataclass
class W12Tensor:
    """A W12 tensor in device memory (all arrays are torch CUDA tensors)."""
    N: int
    K: int
    hi: torch.Tensor       # uint8 [Np*Kp]
    lo: torch.Tensor       # uint8 [Np*Kp/2]
    base: torch.Tensor     # uint8 [N]
    esc_ptr: torch.Tensor  # int32 [Np/16 * groups(K) + 1]
    esc: torch.Tensor      # int32 [esc_cap] (bit pattern of key<<16 | BF16 bits)
    n_esc: int

    @property
    def esc_cap(self) -> int:
        return self.esc.numel()

    def struct(self) -> _Tensor:
        """The C view of the tensor, cached while the same array objects and
        shape are in place (n_esc is refreshed on every call); arrays must not
        be re-pointed in place (Tensor.set_)."""
        c = self.__dict__.get("_cview")
        if (c is None or c[0] is not self.hi or c[1] is not self.lo or c[2] is not self.base
                or c[3] is not self.esc_ptr or c[4] is not self.esc or c[5] != (self.N, self.K)):
            s = _Tensor(self.N, self.K, self.hi.data_ptr(), self.lo.data_ptr(), self.base.data_ptr(),
                        self.esc_ptr.data_ptr(), self.esc.data_ptr(), self.esc_cap, self.n_esc)
            c = (self.hi, self.lo, self.base, self.esc_ptr, self.esc, (self.N, self.K), s)
            self.__dict__["_cview"] = c
        s = c[6]
        s.n_esc = self.n_esc
        return s

    def nbytes(self) -> int:
        """Bytes the tensor stores (all of which the GEMM reads): both
        planes, bases, group offsets and escape entries."""
        return self.hi.numel() + self.lo.numel() + self.N + 4 * self.esc_ptr.numel() + 4 * self.n_esc

    def bits_per_weight(self) -> float:
        return 8.0 * self.nbytes() / max(1, self.N * self.K)

    def rows(self, n0: int, n1: int) -> "W12Tensor":
        """Rows [n0, n1) as a W12 tensor of their own (n0 a multiple of 16):
        plane tiles, bases and the stripes' escape entries are sliced, the
        group offsets rebased (a fresh device tensor)."""
        assert 0 <= n0 <= n1 <= self.N and n0 % 16 == 0
        KT = cols_padded(self.K) // 64
        G = groups(self.K)
        t0, t1 = n0 // 16, (n1 + 15) // 16
        ptr = self.esc_ptr[t0 * G:t1 * G + 1]
        e0 = int(ptr[0].item())
        e1 = int(ptr[-1].item())
        return W12Tensor(n1 - n0, self.K, self.hi[t0 * KT * 1024:t1 * KT * 1024],
                         self.lo[t0 * KT * 512:t1 * KT * 512], self.base[n0:n1], (ptr - e0).contiguous(),
                         self.esc[e0:e1], e1 - e0)


def rows_padded(N: int) -> int:
    return int(load().w12_rows_padded(N))


def groups(K: int) -> int:
    return int(load().w12_groups(K))


def cols_padded(K: int) -> int:
    return int(load().w12_cols_padded(K))


_array_sizes: dict = {}


def _sizes_of(N: int, K: int):
    """(hi bytes, lo bytes, esc_ptr entries) from the library's size queries,
    kept per shape."""
    key = (N, K)
    v = _array_sizes.get(key)
    if v is None:
        lib = load()
        v = (int(lib.w12_hi_bytes(N, K)), int(lib.w12_lo_bytes(N, K)), int(lib.w12_esc_ptr_len(N, K)))
        _array_sizes[key] = v
    return v


def empty_tensor(N: int, K: int, esc_cap: int, device) -> W12Tensor:
    """An uninitialised W12 tensor: one device allocation, the five arrays
    carved out of it at 256-byte aligned offsets."""
    hb, lb, pl = _sizes_of(N, K)
    a = lambda x: (x + 255) & ~255
    o_lo = a(hb)
    o_base = o_lo + a(lb)
    o_ptr = o_base + a(N)
    o_esc = o_ptr + a(4 * pl)
    buf = torch.empty(max(1, o_esc + 4 * esc_cap), dtype=torch.uint8, device=device)
    return W12Tensor(N, K, buf[:hb], buf[o_lo:o_lo + lb], buf[o_base:o_base + N],
                     buf[o_ptr:o_ptr + 4 * pl].view(torch.int32), buf[o_esc:o_esc + 4 * esc_cap].view(torch.int32), 0)


def w12_encode(W: torch.Tensor, esc_cap: int | None = None, stream=None, out: W12Tensor | None = None) -> W12Tensor:
    """BF16 [N,K] (CUDA) -> W12Tensor.  Grows the escape arrays if needed.
    With `out` (a W12Tensor of the same N, K, e.g. from empty_tensor), encodes
    into its buffers instead of allocating; its escape array keeps its
    capacity (entries past n_esc are unused), and a tensor needing more
    escapes than it holds raises W12Error(W12_ERR_CAPACITY)."""
    _need_cuda(W, "W", torch.bfloat16)
    assert W.dim() == 2 and W.stride(1) == 1
    N, K = W.shape
    lib = load()
    if out is not None:
        if (out.N, out.K) != (N, K):
            raise ValueError(f"out is {out.N}x{out.K}, W is {N}x{K}")
        s = out.struct()
        st = lib.w12_encode(ctypes.c_void_p(W.data_ptr()), W.stride(0), ctypes.byref(s), _stream(stream))
        out.n_esc = s.n_esc
        _check(st, "w12_encode")
        return out
    if esc_cap is None:
        esc_cap = max(1024, (N * K) // 256)
    for _ in range(2):
        t = empty_tensor(N, K, esc_cap, W.device)
        s = t.struct()
        st = lib.w12_encode(ctypes.c_void_p(W.data_ptr()), W.stride(0), ctypes.byref(s), _stream(stream))
        t.n_esc = s.n_esc
        if st == W12_ERR_CAPACITY:
            esc_cap = s.n_esc
            continue
        _check(st, "w12_encode")
        t.esc = t.esc[:t.n_esc]
        return t
    raise W12Error(W12_ERR_CAPACITY, "w12_encode")


def w12_decode(t: W12Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(t.N, t.K, dtype=torch.bfloat16, device=t.hi.device)
    _need_cuda(out, "out", torch.bfloat16)
    s = t.struct()
    _check(load().w12_decode(ctypes.byref(s), ctypes.c_void_p(out.data_ptr()), out.stride(0) if t.K else t.K,
                             _stream(stream)), "w12_decode")
    return out


_ws_cache: dict = {}


def verify_workspace(device) -> torch.Tensor:
    key = ("verify", torch.device(device))
    if key not in _ws_cache:
        _ws_cache[key] = torch.zeros(int(load().w12_verify_workspace_bytes()), dtype=torch.uint8, device=device)
    return _ws_cache[key]


def w12_verify_roundtrip(W: torch.Tensor, t: W12Tensor, workspace: torch.Tensor | None = None, stream=None):
    """Bitwise load-time check.  Returns (status, n_mismatch); status is
    W12_OK, W12_ERR_MISMATCH or W12_ERR_CORRUPT (other errors raise)."""
    _need_cuda(W, "W", torch.bfloat16)
    ws = workspace if workspace is not None else verify_workspace(W.device)
    s = t.struct()
    nm = ctypes.c_int64(0)
    st = load().w12_verify_roundtrip(ctypes.c_void_p(W.data_ptr()), W.stride(0) if t.K else t.K, ctypes.byref(s),
                                     ctypes.byref(nm), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                     _stream(stream))
    if st not in (W12_OK, W12_ERR_MISMATCH, W12_ERR_CORRUPT):
        _check(st, "w12_verify_roundtrip")
    return st, nm.value


def make_opts(max_ctas=0, split_k=0, path=W12_PATH_AUTO, flags=0) -> GemmOpts:
    return GemmOpts(max_ctas, split_k, path, flags)


def w12_gemm_workspace_bytes(M: int, N: int, K: int, opts: GemmOpts | None = None) -> int:
    o = opts if opts is not None else make_opts()
    return int(load().w12_gemm_workspace_bytes(M, N, K, ctypes.byref(o)))


class Workspace:
    """A zero-filled device workspace that grows on demand (torch-allocated)."""

    def __init__(self, device, nbytes: int = 0):
        self.device = torch.device(device)
        self.buf = torch.zeros(max(256, nbytes), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


def default_workspace(device) -> Workspace:
    key = ("gemm", torch.device(device))
    if key not in _ws_cache:
        _ws_cache[key] = Workspace(device)
    return _ws_cache[key]


def w12_gemm(A: torch.Tensor, t: W12Tensor, Y: torch.Tensor | None = None, workspace: Workspace | None = None,
             opts: GemmOpts | None = None, stream=None) -> torch.Tensor:
    """Y[M,N] = A[M,K] * W^T with W in W12 (BF16 out, FP32 accumulation)."""
    o = opts if opts is not None else make_opts()
    _check_gemm_operands(A, t, Y, o.flags)
    M = A.shape[0]
    if Y is None:
        Y = torch.empty(M, _out_cols(t, o.flags), dtype=torch.bfloat16, device=A.device)
    need = w12_gemm_workspace_bytes(M, t.N, t.K, o)
    ws = (workspace or default_workspace(A.device)).ensure(max(need, 256))
    s = t.struct()
    _check(load().w12_gemm(ctypes.c_void_p(A.data_ptr()), A.stride(0), ctypes.byref(s),
                           ctypes.c_void_p(Y.data_ptr()), Y.stride(0), M, ctypes.c_void_p(ws.data_ptr()),
                           ws.numel(), ctypes.byref(o), _stream(stream)), "w12_gemm")
    return Y


class GemmCall:
    """w12_gemm with every argument marshalled once (for launch loops and
    benchmarks): calling the object only invokes the C entry point."""

    def __init__(self, A: torch.Tensor, t: W12Tensor, Y: torch.Tensor, workspace: Workspace,
                 opts: GemmOpts | None = None, stream=None):
        self._opts = opts if opts is not None else make_opts()
        _check_gemm_operands(A, t, Y, self._opts.flags)
        need = w12_gemm_workspace_bytes(A.shape[0], t.N, t.K, self._opts)
        ws = workspace.ensure(max(need, 256))
        self._keep = (A, t, Y, ws)  # the buffer itself: a later ensure() may replace it
        self._struct = t.struct()
        self._fn = load().w12_gemm
        self._args = (ctypes.c_void_p(A.data_ptr()), A.stride(0), ctypes.byref(self._struct),
                      ctypes.c_void_p(Y.data_ptr()), Y.stride(0), A.shape[0], ctypes.c_void_p(ws.data_ptr()),
                      ws.numel(), ctypes.byref(self._opts), _stream(stream))

    def __call__(self):
        st = self._fn(*self._args)
        if st != W12_OK:
            raise W12Error(st, "w12_gemm")


class GemmListCall:
    """w12_gemm_list with every argument marshalled once: calling the object
    only invokes the C entry point.  entries: a sequence of (A, t, Y, after,
    flags) with A [M, K] and Y [M, N] (or [M, N/2] with W12_GEMM_SILU_MUL)
    CUDA bfloat16 tensors, t a W12Tensor, after -1 or the index of an earlier
    entry whose output this entry's A depends on."""

    def __init__(self, entries, workspace: Workspace, opts: GemmOpts | None = None, stream=None):
        self._opts = opts if opts is not None else make_opts()
        n = len(entries)
        self._structs = []
        items = (GemmItem * max(1, n))()
        for i, (A, t, Y, after, flags) in enumerate(entries):
            _check_gemm_operands(A, t, Y, flags)
            if not -1 <= after < i:
                raise ValueError(f"entry {i}: after must be -1 or an earlier entry, got {after}")
            st = t.struct()
            self._structs.append(st)
            items[i] = GemmItem(A.data_ptr(), A.stride(0), ctypes.pointer(st), Y.data_ptr(), Y.stride(0),
                                A.shape[0], after, flags)
        self._items = items
        need = int(load().w12_gemm_list_workspace_bytes(items, n, ctypes.byref(self._opts)))
        if n and need == 0:
            raise W12Error(W12_ERR_INVALID, "w12_gemm_list_workspace_bytes")
        ws = workspace.ensure(max(need, 256))
        self._keep = (entries, ws)
        self._fn = load().w12_gemm_list
        self._args = (items, n, ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(self._opts),
                      _stream(stream))

    def __call__(self):
        st = self._fn(*self._args)
        if st != W12_OK:
            raise W12Error(st, "w12_gemm_list")


def w12_gemm_list(entries, workspace: Workspace | None = None, opts: GemmOpts | None = None, stream=None):
    """Several small-M GEMMs in one persistent launch (w12_gemm_list); see
    GemmListCall.  Returns the outputs."""
    ws = workspace or default_workspace(entries[0][0].device if entries else "cuda")
    GemmListCall(entries, ws, opts, stream)()
    return [e[2] for e in entries]


def w12_gemm_noalloc(A: torch.Tensor, t: W12Tensor, Y: torch.Tensor, opts: GemmOpts | None = None,
                     stream=None) -> torch.Tensor:
    """w12_gemm without a workspace: the library's built-in scratch array is
    used (for callers that cannot allocate device memory).  Y must be given."""
    if Y is None:
        raise ValueError("w12_gemm_noalloc needs the output Y")
    o = opts if opts is not None else make_opts()
    _check_gemm_operands(A, t, Y, o.flags)
    s = t.struct()
    _check(load().w12_gemm_noalloc(ctypes.c_void_p(A.data_ptr()), A.stride(0), ctypes.byref(s),
                                   ctypes.c_void_p(Y.data_ptr()), Y.stride(0), A.shape[0], ctypes.byref(o),
                                   _stream(stream)), "w12_gemm_noalloc")
    return Y


W12_TREE_MAX_DEPTH = 16
W12_TREE_MAX_CANDIDATES = 16
W12_TREE_MAX_BUDGET = 256
W12_GDN_PATH = 0
W12_GDN_WY = 1
W12_GDN_MAX_DEPTH = 16
W12_GDN_MAX_NODES = 1024
W12_GDN_MAX_REQUESTS = 65536


class TreeCall:
    """w12_tree_select with its outputs and workspace allocated and every
    argument marshalled once: calling the object only invokes the C entry
    point.  lp: CUDA float32 [R, D, C] log-probabilities (read at each call).
    Outputs (device): req, depth, path (int64 holding the uint64 bits), score,
    parent ([budget] when shared, else [R, budget]) and count ([1] or [R])."""

    def __init__(self, lp: torch.Tensor, budget: int, shared: bool, stream=None):
        if not (lp.is_cuda and lp.dtype == torch.float32 and lp.dim() == 3 and lp.is_contiguous()):
            raise ValueError("lp must be a contiguous CUDA float32 [R, D, C] tensor")
        R, D, C = lp.shape
        n = budget if shared else R * budget
        dev = lp.device
        self.out = {"req": torch.empty(n, dtype=torch.int32, device=dev),
                    "depth": torch.empty(n, dtype=torch.int32, device=dev),
                    "path": torch.empty(n, dtype=torch.int64, device=dev),
                    "score": torch.empty(n, dtype=torch.float32, device=dev),
                    "parent": torch.empty(n, dtype=torch.int32, device=dev),
                    "count": torch.empty(1 if shared else R, dtype=torch.int32, device=dev)}
        need = int(load().w12_tree_workspace_bytes(R, budget))
        self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self._keep = lp
        self._fn = load().w12_tree_select
        self._args = (ctypes.c_void_p(lp.data_ptr()), R, D, C, budget, 1 if shared else 0,
                      *(ctypes.c_void_p(self.out[k].data_ptr())
                        for k in ("req", "depth", "path", "score", "parent", "count")),
                      ctypes.c_void_p(self._ws.data_ptr()), self._ws.numel(), _stream(stream))
        if not shared:
            for k in ("req", "depth", "path", "score", "parent"):
                self.out[k] = self.out[k].view(R, budget)

    def __call__(self) -> dict:
        _check(self._fn(*self._args), "w12_tree_select")
        return self.out


def w12_tree_select(lp: torch.Tensor, budget: int, shared: bool, stream=None) -> dict:
    """Best-first draft-tree node selection (w12_tree_select); see TreeCall."""
    return TreeCall(lp, budget, shared, stream)()


class GdnCall:
    """w12_gdn_tree with its output and workspace allocated and every argument
    marshalled once: calling the object only invokes the C entry point.
    S0: CUDA float32 [R, H, D, D]; q, k, v: CUDA bfloat16 [n, H, D]; alpha,
    beta: CUDA float32 [n, H]; parent: CUDA int32 [n]; req: CUDA int32 [n] or
    None.  mode: W12_GDN_PATH or W12_GDN_WY.  Output `out`: float32 [n, H, D]."""

    def __init__(self, S0, q, k, v, alpha, beta, parent, req=None, mode=None, stream=None):
        mode = W12_GDN_WY if mode is None else mode
        if not (S0.is_cuda and S0.dtype == torch.float32 and S0.dim() == 4 and S0.is_contiguous()):
            raise ValueError("S0 must be a contiguous CUDA float32 [R, H, D, D] tensor")
        R, H, D, D2 = S0.shape
        if D2 != D:
            raise ValueError("S0 must be square per head")
        n = q.shape[0]
        for name, x, shape, dt in (("q", q, (n, H, D), torch.bfloat16), ("k", k, (n, H, D), torch.bfloat16),
                                   ("v", v, (n, H, D), torch.bfloat16), ("alpha", alpha, (n, H), torch.float32),
                                   ("beta", beta, (n, H), torch.float32), ("parent", parent, (n,), torch.int32)):
            if not (x.is_cuda and x.dtype == dt and tuple(x.shape) == shape and x.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor of shape {shape}")
        if req is not None and not (req.is_cuda and req.dtype == torch.int32 and tuple(req.shape) == (n,)
                                    and req.is_contiguous()):
            raise ValueError("req must be a contiguous CUDA int32 [n] tensor or None")
        self.out = torch.empty(n, H, D, dtype=torch.float32, device=q.device)
        need = int(load().w12_gdn_workspace_bytes(n, H, D, mode))
        if need == 0:
            raise W12Error(W12_ERR_INVALID, "w12_gdn_workspace_bytes")
        self._ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        self._keep = (S0, q, k, v, alpha, beta, parent, req)
        self._fn = load().w12_gdn_tree
        ptr = lambda x: ctypes.c_void_p(x.data_ptr() if x is not None else None)  # noqa: E731
        self._args = (ptr(S0), ptr(q), ptr(k), ptr(v), ptr(alpha), ptr(beta), ptr(parent), ptr(req),
                      n, H, R, D, ptr(self.out), ptr(self._ws), self._ws.numel(), mode, _stream(stream))
        self._stream = stream

    def __call__(self) -> torch.Tensor:
        _check(self._fn(*self._args), "w12_gdn_tree")
        return self.out

    def status(self) -> int:
        """The device-side tree check of the last call (synchronous)."""
        return load().w12_gdn_status(ctypes.c_void_p(self._ws.data_ptr()), self._ws.numel(), _stream(self._stream))


def w12_gdn_tree(S0, q, k, v, alpha, beta, parent, req=None, mode=None, stream=None) -> torch.Tensor:
    """Gated-delta-rule outputs of draft-tree nodes (w12_gdn_tree); see GdnCall."""
    return GdnCall(S0, q, k, v, alpha, beta, parent, req, mode, stream)()


def w12_gemm_noalloc_status(stream=None) -> int:
    """W12_ERR_TIMEOUT if a bounded wait of the last w12_gemm_noalloc call on
    the current device gave up (read and cleared; synchronous), else W12_OK."""
    return load().w12_gemm_noalloc_status(_stream(stream))


def w12_gemm_workspace_status(workspace: Workspace, stream=None) -> int:
    return load().w12_gemm_workspace_status(ctypes.c_void_p(workspace.buf.data_ptr()), workspace.buf.numel(),
                                            _stream(stream))
