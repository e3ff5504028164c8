"""The C-ABI library loads, exports every symbol include/w12.h declares, and
its host-side argument checks reject bad calls before touching the GPU."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"\b(w12_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("w12_encode", "w12_decode", "w12_gemm", "w12_verify_roundtrip"):
        assert n in names


def test_library_exports_every_declared_symbol(w12lib):
    lib = ctypes.CDLL(w12lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(w12lib.EXPORTS)


def test_size_queries(w12lib):
    lib = w12lib.load()
    assert lib.w12_rows_padded(5121) == 5136
    assert lib.w12_cols_padded(17400) == 17408
    assert lib.w12_hi_bytes(5121, 17400) == 5136 * 17408
    assert lib.w12_lo_bytes(5121, 17400) == 5136 * 17408 // 2
    assert lib.w12_rows_padded(-1) == -1
    assert lib.w12_verify_workspace_bytes() == 16
    assert lib.w12_groups(5120) == 20 and lib.w12_groups(17400) == 68 and lib.w12_groups(65) == 1
    assert lib.w12_cols_padded(65) == 256 and lib.w12_cols_padded(1000) == 1024
    assert lib.w12_esc_ptr_len(5121, 17400) == 321 * 68 + 1
    assert (lib.w12_version() >> 16) == 1


def test_oracle_and_library_agree_on_sizes(w12lib, oracle):
    lib = w12lib.load()
    for N, K in ((1, 1), (16, 64), (17, 65), (5121, 17400), (34816, 5120), (3, 300)):
        assert w12lib.rows_padded(N) == oracle.rows_padded(N)
        assert w12lib.cols_padded(K) == oracle.cols_padded(K)
        assert lib.w12_groups(K) == oracle.groups(K)
        assert lib.w12_esc_ptr_len(N, K) == oracle.ptr_len(N, K)


def test_gemm_workspace_query(w12lib):
    o = w12lib.make_opts()
    base = 256 + 4 * 65536  # error word + arrival counters
    T, G = 5120 // 16, 5120 // 256
    # small-M path: FP32 partial slots of [16 rows, MP tokens], MP = 8 (M <= 8) or 16 (M <= 16);
    # the automatic cut has at most two partial pieces per range and one range per unit
    for M, mp in ((1, 8), (16, 16)):
        slots, rem = divmod(w12lib.w12_gemm_workspace_bytes(M, 5120, 5120, o) - base, 16 * mp * 4)
        assert rem == 0 and 0 < slots <= 2 * T * G
    # a forced split of S K-chunks per stripe: one slot per (stripe, chunk)
    assert w12lib.w12_gemm_workspace_bytes(1, 5120, 5120, w12lib.make_opts(split_k=4)) == base + T * 4 * 16 * 8 * 4
    assert w12lib.w12_gemm_workspace_bytes(1, 5120, 5120, w12lib.make_opts(split_k=1)) == 256
    assert w12lib.w12_gemm_workspace_bytes(17, 64, 64, w12lib.make_opts(path=w12lib.W12_PATH_MMA)) == 0
    assert w12lib.w12_gemm_workspace_bytes(257, 64, 64, o) == 0  # beyond the tensor-core path
    # the tensor-core path keeps [S][Mpad][Np] partials
    nb = w12lib.w12_gemm_workspace_bytes(40, 1024, 4096, o)
    S, rem = divmod(nb - 256 - 4 * 65536, 48 * 1024 * 4)
    assert rem == 0 and S >= 2
    bad = w12lib.GemmOpts(0, 0, 0, 8)  # unknown flag bit
    assert w12lib.w12_gemm_workspace_bytes(1, 64, 64, bad) == 0


def tc_split(w12lib, M, N, K, opts=None):
    """The tensor-core split S, read back from the workspace size ([S][Mpad][Np] FP32 partials)."""
    nb = w12lib.w12_gemm_workspace_bytes(M, N, K, opts or w12lib.make_opts())
    if nb == 256:
        return 1
    mp, np_ = (M + 15) // 16 * 16, (N + 15) // 16 * 16
    S, rem = divmod(nb - 256 - 4 * 65536, mp * np_ * 4)
    assert rem == 0
    return S


@pytest.mark.parametrize("M,N,K,S", [
    (24, 7168, 5120, 5),    # 56 row tiles x 5 = 280 CTAs: two CTAs per SM
    (64, 7168, 5120, 5),
    (128, 7168, 5120, 2),   # 56 x 4 (partial-traffic cap 4) = 224 < 258: one CTA per SM, 152/56 = 2
    (256, 5120, 5120, 3),   # Mpad > 128: 152/40 = 3 (cap 0.15*5120/256 = 3; 0.1 would give 2)
    (128, 5120, 2048, 1),   # cap 1.6
    (64, 34816, 5120, 1),   # 272 row tiles fill two CTAs per SM without a split
    (24, 5120, 17408, 7),   # 40 x 7 = 280
    (128, 5120, 17408, 7),
    (144, 5120, 8192, 3),   # Mpad > 128 never takes two CTAs per SM (40 x 32 units: too few for ranges)
    (24, 1024, 5120, 16),   # 8 row tiles: at most 16 chunks
    (24, 1024, 1024, 3),    # cap 3.2 (below the 4 column groups whenever Mpad > 25.6)
])
def test_tc_split_rule(M, N, K, S, w12lib):
    """The split (and with it the build) depends on (M, N, K) only: S chunks over 2 x 152
    slots when that grid has >= 258 CTAs and Mpad <= 128, else over 152 slots; each
    capped by the column groups, 16, and the partial traffic 0.1*K/Mpad (0.15*K/Mpad above
    Mpad = 128)."""
    assert tc_split(w12lib, M, N, K) == S


@pytest.mark.parametrize("M,N,K", [
    (256, 34816, 5120),   # 272 row tiles x 20 groups = 5440 units
    (256, 5120, 17408),   # 40 x 68 = 2720
    (144, 5120, 17408),
    (136, 9728, 8192),    # 76 x 32 = 2432 = 16 x 152: the smallest such grid
])
def test_tc_balanced_ranges_plan(M, N, K, w12lib):
    """Mpad > 128 and at least 16 (row tile, group) units per SM: 152 balanced ranges, two FP32
    slots of [Mpad][128] each (a range's first and last piece), instead of K-chunks."""
    mp = (M + 15) // 16 * 16
    assert w12lib.w12_gemm_workspace_bytes(M, N, K, w12lib.make_opts()) == 256 + 4 * 65536 + 2 * 152 * mp * 128 * 4


def test_tc_balanced_ranges_not_taken(w12lib):
    # fewer than 16 units per SM (76 x 31 = 2356), Mpad <= 128, or a forced split: K-chunks
    assert tc_split(w12lib, 136, 9728, 7936) == 2  # 152/76 = 2 chunks
    assert tc_split(w12lib, 128, 9728, 8192) == 4  # Mpad <= 128: 76 row tiles x 4 = 304 CTAs, two per SM
    assert tc_split(w12lib, 256, 34816, 5120, w12lib.make_opts(split_k=2)) == 2


def test_tc_split_at_most_one_chunk_per_group(w12lib):
    # Mpad = 16 (the tensor-core path forced at M <= 16): cap 6.4, 4 column groups
    assert tc_split(w12lib, 16, 1024, 1024, w12lib.make_opts(path=w12lib.W12_PATH_TC)) == 4


def test_noalloc_scratch_holds_every_small_m_plan(w12lib):
    """w12_gemm_noalloc promises that the automatic plan of every shape with
    M <= 16 fits its built-in scratch; the automatic tensor-core plan of a
    5120 x 5120 layer at M = 17 does not."""
    from lossless_bit_weight_02_gb300 import synth
    cap = w12lib.W12_NOALLOC_SCRATCH_BYTES
    shapes = [(N, K) for _, N, K in synth.LAYER_SHAPES]
    shapes += [(5121, 17400), (1, 1), (77829, 256), (16, 1 << 20)]
    for N, K in shapes:
        for M in range(1, 17):
            nb = w12lib.w12_gemm_workspace_bytes(M, N, K)
            assert 0 < nb <= cap, (M, N, K, nb)
    assert w12lib.w12_gemm_workspace_bytes(17, 5120, 5120) > cap
    # with split_k = 1 forced, the tensor-core path needs no partials at any M
    for M in (17, 64, 256):
        assert w12lib.w12_gemm_workspace_bytes(M, 34816, 5120, w12lib.make_opts(split_k=1)) == 256


def test_noalloc_host_side_statuses(w12lib):
    """w12_gemm_noalloc returns w12_gemm's status for options w12_gemm rejects,
    and W12_ERR_CAPACITY for work beyond its scratch, before any CUDA call."""
    lib = w12lib.load()
    t = w12lib._Tensor(5120, 5120, 256, 512, 768, 1024, 1280, 1, 0)
    mma = w12lib.make_opts(path=w12lib.W12_PATH_MMA)
    st = lib.w12_gemm_noalloc(ctypes.c_void_p(4096), 5120, ctypes.byref(t), ctypes.c_void_p(8192), 5120, 17,
                              ctypes.byref(mma), None)
    assert st == w12lib.W12_ERR_UNSUPPORTED
    st = lib.w12_gemm_noalloc(ctypes.c_void_p(4096), 5120, ctypes.byref(t), ctypes.c_void_p(8192), 5120, 17,
                              None, None)
    assert st == w12lib.W12_ERR_CAPACITY
    bad = w12lib.GemmOpts(0, 0, 0, 8)  # unknown flag bit
    st = lib.w12_gemm_noalloc(ctypes.c_void_p(4096), 5120, ctypes.byref(t), ctypes.c_void_p(8192), 5120, 1,
                              ctypes.byref(bad), None)
    assert st == w12lib.W12_ERR_INVALID


def test_status_strings(w12lib):
    for code, name in ((0, "W12_OK"), (-3, "W12_ERR_CAPACITY"), (-7, "W12_ERR_CORRUPT")):
        assert w12lib.status_string(code) == name


def test_invalid_arguments_rejected_on_host(w12lib):
    """These calls fail validation before any CUDA call is made."""
    lib = w12lib.load()
    T = w12lib._Tensor
    t = T(4, 64, None, None, None, None, None, 0, 0)
    assert lib.w12_decode(ctypes.byref(t), None, 64, None) == w12lib.W12_ERR_INVALID
    assert lib.w12_encode(None, 64, None, None) == w12lib.W12_ERR_INVALID
    neg = T(-1, 64, None, None, None, None, None, 0, 0)
    assert lib.w12_decode(ctypes.byref(neg), None, 64, None) == w12lib.W12_ERR_INVALID
    # misaligned planes
    good = T(4, 64, 16, 17, 32, 48, 64, 1, 0)
    assert lib.w12_decode(ctypes.byref(good), ctypes.c_void_p(4096), 64, None) == w12lib.W12_ERR_ALIGN
    # M > 16 on the mma path
    t2 = T(16, 64, 256, 512, 768, 1024, 1280, 1, 0)
    o = w12lib.make_opts(path=w12lib.W12_PATH_MMA)
    st = lib.w12_gemm(ctypes.c_void_p(4096), 64, ctypes.byref(t2), ctypes.c_void_p(8192), 16, 17,
                      ctypes.c_void_p(16384), 1 << 20, ctypes.byref(o), None)
    assert st == w12lib.W12_ERR_UNSUPPORTED
    # lda not a multiple of 8
    st = lib.w12_gemm(ctypes.c_void_p(4096), 65, ctypes.byref(t2), ctypes.c_void_p(8192), 16, 1,
                      ctypes.c_void_p(16384), 1 << 20, None, None)
    assert st == w12lib.W12_ERR_ALIGN
    # workspace too small
    st = lib.w12_gemm(ctypes.c_void_p(4096), 64, ctypes.byref(t2), ctypes.c_void_p(8192), 16, 1,
                      ctypes.c_void_p(16384), 8, None, None)
    assert st == w12lib.W12_ERR_CAPACITY
    nm = ctypes.c_int64()
    st = lib.w12_verify_roundtrip(ctypes.c_void_p(4096), 64, ctypes.byref(t2), ctypes.byref(nm),
                                  ctypes.c_void_p(16384), 4, None)
    assert st == w12lib.W12_ERR_CAPACITY


def test_tree_select_argument_checks(w12lib):
    """Host-side validation of w12_tree_select: nothing is launched (no GPU needed)."""
    lib = w12lib.load()
    assert lib.w12_tree_workspace_bytes(0, 8) == 0 and lib.w12_tree_workspace_bytes(4, 257) == 0
    assert lib.w12_tree_workspace_bytes(64, 63) > 0
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation
    args = [p] * 6 + [p, ctypes.c_size_t(1 << 30), None]
    for R, D, C, B, shared in ((0, 8, 8, 32, 0), (4, 0, 8, 32, 0), (4, 17, 8, 32, 0), (4, 8, 17, 32, 0),
                               (4, 8, 8, 0, 0), (4, 8, 8, 257, 1), (4, 8, 8, 32, 2)):
        assert lib.w12_tree_select(p, R, D, C, B, shared, *args) == w12lib.W12_ERR_INVALID
    assert lib.w12_tree_select(None, 4, 8, 8, 32, 0, *args) == w12lib.W12_ERR_INVALID
    odd = ctypes.c_void_p((1 << 20) + 4)  # path must be 8-byte aligned
    assert lib.w12_tree_select(p, 4, 8, 8, 32, 0, p, p, odd, p, p, p, p, ctypes.c_size_t(1 << 30),
                               None) == w12lib.W12_ERR_ALIGN
    small = ctypes.c_size_t(lib.w12_tree_workspace_bytes(4, 32) - 1)
    assert lib.w12_tree_select(p, 4, 8, 8, 32, 0, p, p, p, p, p, p, p, small, None) == w12lib.W12_ERR_CAPACITY


def test_gdn_argument_checks(w12lib):
    """Host-side validation of w12_gdn_tree: nothing is launched (no GPU needed)."""
    lib = w12lib.load()
    PATH, WY = w12lib.W12_GDN_PATH, w12lib.W12_GDN_WY
    assert lib.w12_gdn_workspace_bytes(63, 32, 128, PATH) == 256
    assert lib.w12_gdn_workspace_bytes(63, 32, 128, WY) == 256 + 2 * 63 * 32 * 128 * 4 + (63 * 17 * 4 + 15) // 16 * 16
    for n, H, D, mode in ((-1, 4, 64, WY), (1025, 4, 64, WY), (8, 0, 64, WY), (8, 4, 96, WY), (8, 4, 64, 2)):
        assert lib.w12_gdn_workspace_bytes(n, H, D, mode) == 0
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation
    big = ctypes.c_size_t(1 << 30)

    def call(*ptrs, n=8, H=4, R=1, D=64, ws=big, mode=WY):
        return lib.w12_gdn_tree(*ptrs[:8], n, H, R, D, ptrs[8], ptrs[9], ws, mode, None)

    ok = [p] * 10
    for kw in ({"n": -1}, {"n": 1025}, {"H": 0}, {"R": 0}, {"R": w12lib.W12_GDN_MAX_REQUESTS + 1}, {"D": 32},
               {"D": 100}, {"mode": 3}):
        assert call(*ok, **kw) == w12lib.W12_ERR_INVALID, kw
    for i in range(10):
        if i == 7:  # req may be NULL
            continue
        ptrs = list(ok)
        ptrs[i] = None
        assert call(*ptrs) == w12lib.W12_ERR_INVALID, i
    for i, off in ((0, 4), (1, 2), (3, 8), (4, 2), (6, 1), (7, 2), (8, 4), (9, 8)):
        ptrs = list(ok)
        ptrs[i] = ctypes.c_void_p((1 << 20) + off)
        assert call(*ptrs) == w12lib.W12_ERR_ALIGN, i
    need = lib.w12_gdn_workspace_bytes(8, 4, 64, WY)
    assert call(*ok, ws=ctypes.c_size_t(need - 1)) == w12lib.W12_ERR_CAPACITY
    assert lib.w12_gdn_status(None, 256, None) == w12lib.W12_ERR_INVALID
    assert lib.w12_gdn_status(p, 255, None) == w12lib.W12_ERR_INVALID


def test_empty_tensor_is_one_allocation_with_aligned_arrays(w12lib):
    """empty_tensor carves the five arrays out of one buffer: sizes as the
    library's size queries give them, every array at a 256-byte aligned offset
    (the planes are read by TMA, which wants 16-byte aligned addresses)."""
    lib = w12lib.load()
    for N, K, cap in ((0, 64, 1024), (5, 0, 10), (17, 65, 3), (34816, 5120, 1000), (1, 1, 0)):
        t = w12lib.empty_tensor(N, K, cap, "cpu")
        assert t.hi.numel() == lib.w12_hi_bytes(N, K) and t.lo.numel() == lib.w12_lo_bytes(N, K)
        assert t.base.numel() == N and t.esc_ptr.numel() == lib.w12_esc_ptr_len(N, K)
        assert t.esc.numel() == cap and t.esc.dtype == torch.int32 and t.esc_ptr.dtype == torch.int32
        arrays = (t.hi, t.lo, t.base, t.esc_ptr, t.esc)
        assert all(x.storage_offset() * x.element_size() % 256 == 0 for x in arrays), (N, K)
        assert len({x.untyped_storage().data_ptr() for x in arrays}) == 1
