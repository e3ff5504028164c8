"""GPU encode / decode / verify against the oracle (bit-exact).

SpecPilot (arXiv 2611.02501), section 4.1: W12 is lossless and every decoded
tensor is checked bit for bit at load time.  Here the CUDA encoder must
produce the oracle's bytes exactly (planes, bases, row offsets, escapes), the
CUDA decoder must return the original BF16 bits, and the CUDA verifier must
count exactly the mismatches the oracle counts on host-corrupted tensors.
"""
import ctypes

import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth

pytestmark = pytest.mark.gpu


def host_view(t):
    """A GPU W12Tensor's arrays as numpy (for comparison only)."""
    return dict(
        hi=t.hi.cpu().numpy(), lo=t.lo.cpu().numpy(), base=t.base.cpu().numpy(),
        esc_ptr=t.esc_ptr.cpu().numpy(), esc=t.esc[:t.n_esc].cpu().numpy().view(np.uint32), n_esc=t.n_esc)


def upload(w, ref):
    """An oracle-built (host) W12 tensor copied to the device."""
    dev = "cuda"
    esc = torch.from_numpy(ref.esc.view(np.int32)).to(dev) if ref.esc.size else \
        torch.zeros(0, dtype=torch.int32, device=dev)
    return w.W12Tensor(ref.N, ref.K, torch.from_numpy(ref.hi).to(dev), torch.from_numpy(ref.lo).to(dev),
                       torch.from_numpy(ref.base).to(dev), torch.from_numpy(ref.esc_ptr).to(dev), esc,
                       ref.n_esc)


def single_window_rows(N, K, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(1, 240, size=(N, 1))
    e = b + rng.integers(0, 16, size=(N, K))
    s = rng.integers(0, 2, size=(N, K))
    m = rng.integers(0, 128, size=(N, K))
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


CASES = {
    "dense_1024x1024": lambda: synth.dense_weights(1024, 1024, seed=0),
    "adversarial_200x1000": lambda: synth.adversarial_weights(200, 1000, seed=4),
    "all_patterns_64x1024": lambda: synth.all_patterns(64, seed=0),
    "one_weight": lambda: synth.dense_weights(1, 1, seed=1),
    "ragged_17x65": lambda: synth.dense_weights(17, 65, seed=2),
    "ragged_33x200": lambda: synth.adversarial_weights(33, 200, seed=3),
    "zero_rows": lambda: np.zeros((20, 130), np.uint16),
    "single_window": lambda: single_window_rows(48, 320, seed=5),
    "long_rows_5x17400": lambda: synth.adversarial_weights(5, 17400, seed=6),
    "odd_row_width_9x1001": lambda: synth.dense_weights(9, 1001, seed=7),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_encode_decode_verify_bit_exact(name, w12lib, oracle):
    W = CASES[name]()
    st, ref = oracle.encode(W)
    assert st == oracle.OK
    Wd = synth.bits_to_tensor(W, "cuda")
    t = w12lib.w12_encode(Wd)
    torch.cuda.synchronize()
    g = host_view(t)
    assert g["n_esc"] == ref.n_esc
    for key in ("hi", "lo", "base", "esc_ptr", "esc"):
        assert np.array_equal(g[key], getattr(ref, key)), key
    D = w12lib.w12_decode(t)
    assert np.array_equal(synth.tensor_to_bits(D), W)
    assert w12lib.w12_verify_roundtrip(Wd, t) == (w12lib.W12_OK, 0)


def test_decode_into_strided_output(w12lib, oracle):
    W = synth.dense_weights(40, 300, seed=8)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    out = torch.full((40, 312), -7.0, dtype=torch.bfloat16, device="cuda")
    w12lib.w12_decode(t, out[:, :300])
    assert np.array_equal(synth.tensor_to_bits(out[:, :300]), W)
    assert (out[:, 300:] == -7.0).all()


def test_encode_strided_input(w12lib, oracle):
    W = synth.dense_weights(30, 200, seed=9)
    big = np.zeros((30, 264), np.uint16)
    big[:, :200] = W
    Wd = synth.bits_to_tensor(big, "cuda")[:, :200]
    t = w12lib.w12_encode(Wd)
    st, ref = oracle.encode(W)
    assert np.array_equal(t.hi.cpu().numpy(), ref.hi)
    assert np.array_equal(t.esc.cpu().numpy().view(np.uint32), ref.esc)


def test_encode_capacity_path(w12lib, oracle):
    W = synth.dense_weights(64, 512, seed=10)
    st, full = oracle.encode(W)
    cap = full.n_esc // 2
    assert cap > 1
    lib = w12lib.load()
    t = w12lib.empty_tensor(64, 512, cap, "cuda")
    s = t.struct()
    Wd = synth.bits_to_tensor(W, "cuda")
    rc = lib.w12_encode(ctypes.c_void_p(Wd.data_ptr()), 512, ctypes.byref(s), w12lib._stream())
    torch.cuda.synchronize()
    assert rc == w12lib.W12_ERR_CAPACITY and s.n_esc == full.n_esc
    assert np.array_equal(t.hi.cpu().numpy(), full.hi)
    assert np.array_equal(t.lo.cpu().numpy(), full.lo)
    assert np.array_equal(t.esc_ptr.cpu().numpy(), full.esc_ptr)
    assert np.array_equal(t.esc.cpu().numpy().view(np.uint32), full.esc[:cap])


def test_empty_shapes(w12lib):
    t = w12lib.w12_encode(torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"))
    assert t.n_esc == 0 and t.esc_ptr.cpu().tolist() == [0]
    Wk0 = torch.zeros(5, 0, dtype=torch.bfloat16, device="cuda")
    t = w12lib.w12_encode(Wk0)
    assert t.n_esc == 0 and t.esc_ptr.cpu().tolist() == [0]
    assert (t.base.cpu().numpy() == 239).all()
    assert w12lib.w12_decode(t).shape == (5, 0)
    assert w12lib.w12_verify_roundtrip(Wk0, t) == (w12lib.W12_OK, 0)


def test_verify_counts_host_corruption(w12lib, oracle):
    """Corruption is planted in host copies of the oracle's tensor; the GPU
    verifier must report the oracle's count for each."""
    W = synth.dense_weights(64, 640, seed=11)
    Wd = synth.bits_to_tensor(W, "cuda")
    st, ref = oracle.encode(W)
    rng = np.random.default_rng(12)
    plans = []
    for trial in range(12):
        c = ref.copy()
        kind = trial % 4
        if kind == 0:
            idx = rng.choice(c.hi.size, size=int(rng.integers(1, 40)), replace=False)
            c.hi[idx] ^= rng.integers(1, 256, idx.size).astype(np.uint8)
        elif kind == 1:
            idx = rng.choice(c.lo.size, size=int(rng.integers(1, 40)), replace=False)
            c.lo[idx] ^= rng.integers(1, 256, idx.size).astype(np.uint8)
        elif kind == 2:
            idx = rng.choice(c.N, size=3, replace=False)
            c.base[idx] ^= np.uint8(1 << int(rng.integers(0, 7)))
        else:
            idx = rng.choice(c.n_esc, size=min(5, c.n_esc), replace=False)
            c.esc[idx] ^= np.uint32(0x0040)
        plans.append(c)
    for c in plans:
        want = oracle.verify(W, c)
        got = w12lib.w12_verify_roundtrip(Wd, upload(w12lib, c))
        assert got == want


def test_verify_flags_malformed_escape_list(w12lib, oracle):
    W = synth.dense_weights(32, 512, seed=13)
    Wd = synth.bits_to_tensor(W, "cuda")
    st, ref = oracle.encode(W)
    g = next(i for i in range(ref.esc_ptr.size - 1) if ref.esc_ptr[i + 1] - ref.esc_ptr[i] >= 2)
    c = ref.copy()
    i = c.esc_ptr[g]
    c.esc[i], c.esc[i + 1] = c.esc[i + 1], c.esc[i]  # keys out of order
    assert oracle.verify(W, c) == (oracle.ERR_CORRUPT, -1)
    assert w12lib.w12_verify_roundtrip(Wd, upload(w12lib, c)) == (w12lib.W12_ERR_CORRUPT, -1)
    c = ref.copy()
    c.esc[0] |= np.uint32(0xF000 << 16)  # key >= 4096
    assert oracle.verify(W, c) == (oracle.ERR_CORRUPT, -1)
    assert w12lib.w12_verify_roundtrip(Wd, upload(w12lib, c)) == (w12lib.W12_ERR_CORRUPT, -1)
    c = ref.copy()
    c.esc_ptr[3] = c.esc_ptr[4] + 1  # offsets not monotone
    assert oracle.verify(W, c) == (oracle.ERR_CORRUPT, -1)
    assert w12lib.w12_verify_roundtrip(Wd, upload(w12lib, c)) == (w12lib.W12_ERR_CORRUPT, -1)


def test_verify_counts_moved_escape(w12lib, oracle):
    """An escape key rewritten to name another weight: the oracle's count of
    mismatches, on the GPU too."""
    W = synth.dense_weights(48, 700, seed=16)
    Wd = synth.bits_to_tensor(W, "cuda")
    st, ref = oracle.encode(W)
    rng = np.random.default_rng(17)
    for _ in range(6):
        c = ref.copy()
        e = int(rng.integers(0, c.n_esc))
        key = int(c.esc[e] >> 16)
        new_key = (key & ~0x3F) | int(rng.integers(0, 64))  # another column of the same tile row
        c.esc[e] = np.uint32((new_key << 16) | (int(c.esc[e]) & 0xFFFF))
        want = oracle.verify(W, c)
        assert w12lib.w12_verify_roundtrip(Wd, upload(w12lib, c)) == want


def test_row_slice_is_a_w12_tensor(w12lib, oracle):
    """Rows [n0, n1) of a tensor (n0 a multiple of 16) decode to the same rows:
    the property that lets output channels be split across devices."""
    W = synth.dense_weights(100, 384, seed=14)
    t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"))
    for n0, n1 in ((0, 16), (16, 48), (32, 100), (96, 100)):
        part = t.rows(n0, n1)
        assert np.array_equal(synth.tensor_to_bits(w12lib.w12_decode(part)), W[n0:n1])


def test_full_size_gate_up_encode_matches_oracle_on_sampled_stripes(w12lib, oracle):
    """Full-size gate/up layer (34816 x 5120) encoded on the GPU; sampled
    stripes compared byte for byte with the oracle's encoding of the same
    rows; the whole tensor checked with the GPU verifier."""
    N, K = 34816, 5120
    Wd = synth.dense_weights_device(N, K, seed=1002)
    t = w12lib.w12_encode(Wd)
    assert w12lib.w12_verify_roundtrip(Wd, t) == (w12lib.W12_OK, 0)
    KT, G = K // 64, K // 256
    rng = np.random.default_rng(15)
    for st_ in list(rng.choice(N // 16, size=6, replace=False)) + [N // 16 - 1]:
        rows = slice(16 * st_, 16 * st_ + 16)
        Wh = synth.tensor_to_bits(Wd[rows])
        s, ref = oracle.encode(Wh)
        assert np.array_equal(t.hi[st_ * KT * 1024:(st_ + 1) * KT * 1024].cpu().numpy(), ref.hi)
        assert np.array_equal(t.lo[st_ * KT * 512:(st_ + 1) * KT * 512].cpu().numpy(), ref.lo)
        assert np.array_equal(t.base[rows].cpu().numpy(), ref.base)
        ptr = t.esc_ptr[st_ * G:st_ * G + G + 1].cpu().numpy()
        assert np.array_equal(ptr - ptr[0], ref.esc_ptr)
        assert np.array_equal(t.esc[ptr[0]:ptr[-1]].cpu().numpy().view(np.uint32), ref.esc)


@pytest.mark.parametrize("name,N,K,seed", [(n, N, K, 1000 + i) for i, (n, N, K) in enumerate(synth.LAYER_SHAPES)] +
                         [("stress", 5121, 17400, 4)])
def test_full_size_encode_bytes_match_the_oracle_on_sampled_stripes(name, N, K, seed, w12lib, oracle):
    """The 27B-class layers (and the escape-stress shape) encoded on the GPU
    at full size, so the window kernel and the pack kernel (with its segmented
    offset scan) run their multi-block grids; then sampled 16-row stripes
    (first, last, and random ones) are
    compared byte for byte with the oracle's encoding of the same rows: hi and
    lo planes, bases, group offsets (rebased to the stripe) and escapes."""
    if name == "stress":
        Wd = synth.bits_to_tensor(synth.adversarial_weights(N, K, seed=seed), "cuda")
    else:
        Wd = synth.dense_weights_device(N, K, seed=seed)
    t = w12lib.w12_encode(Wd)
    T = (N + 15) // 16
    rng = np.random.default_rng(seed)
    stripes = sorted({0, T - 1, T // 2, *rng.choice(T, size=3, replace=False).tolist()})
    for s in stripes:
        n0, n1 = 16 * s, min(N, 16 * s + 16)
        got = host_view(t.rows(n0, n1))
        st, ref = oracle.encode(synth.tensor_to_bits(Wd[n0:n1]))
        assert st == oracle.OK
        assert got["n_esc"] == ref.n_esc, (s, got["n_esc"], ref.n_esc)
        assert np.array_equal(got["hi"], ref.hi), s
        assert np.array_equal(got["lo"], ref.lo), s
        assert np.array_equal(got["base"], ref.base), s
        assert np.array_equal(got["esc_ptr"], ref.esc_ptr), s
        assert np.array_equal(got["esc"], ref.esc[:ref.n_esc]), s


def test_encode_where_scan_blocks_redo_their_segments(w12lib, oracle):
    """Random 16-bit patterns (about 15 escapes in 16 weights) over enough
    16-row stripes that each block of the pack kernel's offset scan holds more
    units whose escapes did not fit a warp's staging area than it can list, so
    it re-derives every unit of its segment from W.  The GPU verifier checks
    the whole tensor; sampled stripes equal the oracle's bytes."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 300 * 4 * sms  # > 256 units per scan block at up to 4 blocks per SM
    N, K = 16 * T, 256
    Wd = synth.random_bits_device(N, K, seed=31)
    t = w12lib.w12_encode(Wd)
    assert t.n_esc > N * K // 2
    assert w12lib.w12_verify_roundtrip(Wd, t) == (w12lib.W12_OK, 0)
    rng = np.random.default_rng(32)
    for s in sorted({0, T - 1, T // 2, *rng.choice(T, size=3, replace=False).tolist()}):
        n0, n1 = 16 * s, 16 * s + 16
        got = host_view(t.rows(n0, n1))
        st, ref = oracle.encode(synth.tensor_to_bits(Wd[n0:n1]))
        assert st == oracle.OK and got["n_esc"] == ref.n_esc, s
        for key in ("hi", "lo", "base", "esc_ptr"):
            assert np.array_equal(got[key], getattr(ref, key)), (s, key)
        assert np.array_equal(got["esc"], ref.esc[:ref.n_esc]), s
    del Wd, t
    torch.cuda.empty_cache()


def test_encode_into_preallocated_tensor(w12lib, oracle):
    """w12_encode(W, out=t) reuses t's buffers: two different tensors of the
    same shape encoded one after the other into the same buffers, each equal
    to the oracle's bytes; a tensor that needs more escapes than t holds
    raises W12_ERR_CAPACITY."""
    N, K = 40, 520
    pre = w12lib.empty_tensor(N, K, 4096, "cuda")
    for seed in (21, 22):
        W = synth.adversarial_weights(N, K, seed=seed)
        st, ref = oracle.encode(W)
        t = w12lib.w12_encode(synth.bits_to_tensor(W, "cuda"), out=pre)
        torch.cuda.synchronize()
        assert t is pre and t.n_esc == ref.n_esc
        g = host_view(t)
        for key in ("hi", "lo", "base", "esc_ptr", "esc"):
            assert np.array_equal(g[key], getattr(ref, key)), key
    small = w12lib.empty_tensor(N, K, 8, "cuda")
    with pytest.raises(w12lib.W12Error) as ei:
        w12lib.w12_encode(synth.bits_to_tensor(synth.adversarial_weights(N, K, seed=23), "cuda"), out=small)
    assert ei.value.status == w12lib.W12_ERR_CAPACITY


@pytest.mark.parametrize("N,K,pad", [(37, 1000, 1), (21, 9000, 3), (16, 256, 5), (40, 8200, 0)])
def test_encode_odd_row_strides(N, K, pad, w12lib, oracle):
    """Rows that are not 16-byte aligned (an odd row stride) take the
    bounds-checked loads in the window search and the pack; rows longer than
    8192 columns take the 4-warp window kernel.  Bytes equal the oracle's."""
    W = synth.adversarial_weights(N, K, seed=40 + N + pad)
    big = np.zeros((N, K + pad), np.uint16)
    big[:, :K] = W
    Wd = synth.bits_to_tensor(big, "cuda")[:, :K]
    t = w12lib.w12_encode(Wd)
    torch.cuda.synchronize()
    st, ref = oracle.encode(W)
    g = host_view(t)
    assert g["n_esc"] == ref.n_esc
    for key in ("hi", "lo", "base", "esc_ptr", "esc"):
        assert np.array_equal(g[key], getattr(ref, key)), key


def test_concurrent_encodes_from_two_threads(w12lib, oracle):
    """Two host threads encode different tensors at once, each on a stream of
    its own (the C call runs without the GIL): each gets its own escape-count
    word and cached launch state, and both results equal the oracle's bytes."""
    import threading
    shapes = [(96, 1300, 61), (80, 2100, 62)]
    Ws = [synth.adversarial_weights(N, K, seed=s) for N, K, s in shapes]
    Wds = [synth.bits_to_tensor(W, "cuda") for W in Ws]
    out = [None, None]
    errors = []

    def run(i):
        try:
            st = torch.cuda.Stream()
            for _ in range(20):
                t = w12lib.w12_encode(Wds[i], stream=st)
            st.synchronize()
            out[i] = t
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i, W in enumerate(Ws):
        st, ref = oracle.encode(W)
        g = host_view(out[i])
        assert g["n_esc"] == ref.n_esc
        for key in ("hi", "lo", "base", "esc_ptr"):
            assert np.array_equal(g[key], getattr(ref, key)), (i, key)
        assert np.array_equal(g["esc"], ref.esc[:ref.n_esc]), i
