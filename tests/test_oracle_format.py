"""Pins for the oracle's W12 format arithmetic (CPU only).

Each test checks the oracle against something other than itself: torch's
exact BF16 -> float conversion, brute force over every BF16 bit pattern or
every window base, hand-worked records, closed forms and invariants of the
format of SpecPilot (arXiv 2611.02501), section 4.1.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from lossless_bit_weight_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_value(bits: np.ndarray) -> np.ndarray:
    """BF16 bits -> float64 values through torch (an independent route)."""
    t = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


ALL = np.arange(65536, dtype=np.uint16)
ALL_VALUES = f32_value(ALL)


def test_bf16_to_double_matches_torch(oracle):
    for b in range(0, 65536, 1):
        v = oracle.bf16_to_double(b)
        ref = ALL_VALUES[b]
        if math.isnan(ref):
            assert math.isnan(v)
        else:
            assert v == ref and math.copysign(1, v) == math.copysign(1, ref), hex(b)


def test_bf16_rounding_exact_values_and_ties(oracle):
    # every finite pattern maps to itself (both zeros keep their sign)
    for b in range(65536):
        e = (b >> 7) & 0xFF
        if e == 255:
            continue
        assert oracle.bf16_from_double(ALL_VALUES[b]) == b, hex(b)
    # midpoints between neighbours go to the even mantissa, and a nudge
    # either way picks the nearer neighbour
    for b in range(0, 0x7F7F):
        lo, hi = ALL_VALUES[b], ALL_VALUES[b + 1]
        mid = (lo + hi) / 2.0  # exact in FP64
        want = b if (b & 1) == 0 else b + 1
        assert oracle.bf16_from_double(mid) == want, hex(b)
        assert oracle.bf16_from_double(-mid) == want | 0x8000
        eps = (hi - lo) / 1024.0
        assert oracle.bf16_from_double(mid - eps) == b
        assert oracle.bf16_from_double(mid + eps) == b + 1


def test_bf16_rounding_overflow_underflow_nan(oracle):
    big = ALL_VALUES[0x7F7F]
    ulp = 2.0 ** (127 - 7)
    assert oracle.bf16_from_double(big + ulp / 2) == 0x7F80  # tie rounds to even = 2^128 = Inf
    assert oracle.bf16_from_double(big + ulp / 2 - ulp / 64) == 0x7F7F
    assert oracle.bf16_from_double(-1e300) == 0xFF80
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000      # half the smallest denormal: tie to 0
    assert oracle.bf16_from_double(1.5 * 2.0 ** -133) == 0x0002  # tie between 1 and 2 -> 2
    assert oracle.bf16_from_double(-(2.0 ** -140)) == 0x8000
    assert oracle.bf16_from_double(float("inf")) == 0x7F80
    r = oracle.bf16_from_double(float("nan"))
    assert (r & 0x7F80) == 0x7F80 and (r & 0x7F) != 0


def test_worked_records(oracle):
    with open(os.path.join(GOLDEN, "worked_records.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for bits, base, esc, rec, hi, lo in rows:
        bits, base, esc = int(bits, 16), int(base), int(esc)
        rec, hi, lo = int(rec, 16), int(hi, 16), int(lo, 16)
        assert oracle.is_escape(bits, base) == bool(esc)
        if not esc:
            r = oracle.record(bits, base)
            assert r == rec and r >> 4 == hi and r & 0xF == lo
            assert oracle.decode_record(r, base) == bits


def _expand_window_row(spec: str) -> np.ndarray:
    vals = []
    for item in spec.split():
        e, c = item.split(":")
        e, c = int(e), int(c)
        vals += [(e << 7) | 0x15] * c if e else [0] * c
    return np.array(vals, np.uint16)


def test_worked_windows(oracle):
    with open(os.path.join(GOLDEN, "worked_windows.txt")) as f:
        rows = [l.split(";") for l in f if l.strip() and not l.startswith("#")]
    for want, spec in rows:
        assert oracle.window_base(_expand_window_row(spec)) == int(want), spec


def brute_force_base(row: np.ndarray) -> int:
    """Direct search: count escapes for every base 1..239, keep the largest
    base with the fewest escapes (fewest escapes == most in-window weights)."""
    e = (row.astype(np.int64) >> 7) & 0xFF
    best, best_b = None, None
    for b in range(1, 240):
        inwin = (e >= 1) & (e <= 254) & (e >= b) & (e <= b + 15)
        esc = int(row.size - inwin.sum())
        if best is None or esc <= best:
            best, best_b = esc, b
    return best_b


def test_window_brute_force_tiny_rows(oracle):
    rng = np.random.default_rng(11)
    for trial in range(400):
        K = int(rng.integers(1, 17))
        lo = int(rng.integers(0, 240))
        span = int(rng.integers(1, 40))
        e = rng.integers(lo, min(255, lo + span) + 1, size=K)
        s = rng.integers(0, 2, size=K)
        m = rng.integers(0, 128, size=K)
        row = ((s << 15) | (e << 7) | m).astype(np.uint16)
        assert oracle.window_base(row) == brute_force_base(row), (trial, row)


def test_record_closed_form(oracle):
    """For in-window weights: value == (-1)^s * 2^(base+off-127) * (1+m/128)."""
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 65536, size=20000).astype(np.uint16)
    bases = rng.integers(1, 240, size=bits.size)
    vals = f32_value(bits)
    checked = 0
    for b, base, v in zip(bits, bases, vals):
        b, base = int(b), int(base)
        e = (b >> 7) & 0xFF
        if e == 0 or e == 255 or not (base <= e <= base + 15):
            assert oracle.is_escape(b, base)
            continue
        r = oracle.record(b, base)
        assert 0 <= r < 4096
        s, off, m = r >> 11, (r >> 7) & 0xF, r & 0x7F
        assert 0 <= off <= 15
        assert (-1.0) ** s * 2.0 ** (base + off - 127) * (1 + m / 128.0) == v
        checked += 1
    assert checked > 1000


def test_layout_is_a_bijection(oracle):
    """Every (n,k) of the padded Np x Kp grid owns a distinct hi byte and a
    distinct lo nibble, covering both planes exactly once."""
    N, K = 37, 300
    Np, Kp = oracle.rows_padded(N), oracle.cols_padded(K)
    assert (Np, Kp) == (48, 512)
    hi_seen = np.zeros(Np * Kp, np.int32)
    lo_seen = np.zeros(Np * Kp, np.int32)
    for n in range(Np):
        for k in range(Kp):
            hi_seen[oracle.hi_offset(n, k, Kp)] += 1
            b, s = oracle.lo_position(n, k, Kp)
            assert s in (0, 4)
            lo_seen[2 * b + (s // 4)] += 1
    assert (hi_seen == 1).all() and (lo_seen == 1).all()


def escaped_mask(W, base):
    e = (W.astype(np.int64) >> 7) & 0xFF
    b = base.astype(np.int64)[:, None]
    return (e == 0) | (e == 255) | (e < b) | (e > b + 15)


def check_invariants(oracle, W, t):
    N, K = W.shape
    assert oracle.check_structure(t) == 0
    assert t.esc_ptr[0] == 0 and t.esc_ptr[-1] == t.n_esc
    assert t.esc_ptr.size == (oracle.rows_padded(N) // 16) * oracle.groups(K) + 1
    assert ((t.base >= 1) & (t.base <= 239)).all()
    esc = escaped_mask(W, t.base)
    # the list holds exactly the escaped positions, each once, with its bits
    pos = [t.position(e) for e in range(t.n_esc)]
    assert sorted(pos) == sorted(map(tuple, np.argwhere(esc).tolist()))
    for e, (n, k) in enumerate(pos):
        assert t.esc_val[e] == W[n, k]
        assert t.esc_key[e] == oracle.key(n, k)
    # order: stripe, group, then tile, row, column inside the group
    order = [(n // 16, k // 256, (k % 256) // 64, n % 16, k % 64) for n, k in pos]
    assert order == sorted(order)
    Kp = oracle.cols_padded(K)
    # the nested 8-bit view: the hi byte of an in-window weight is its top 8
    # record bits s|off|m[6:4]
    rng = np.random.default_rng(1)
    for _ in range(300):
        n, k = int(rng.integers(N)), int(rng.integers(K))
        base = int(t.base[n])
        w = int(W[n, k])
        ew = (w >> 7) & 0xFF
        h = t.hi[oracle.hi_offset(n, k, Kp)]
        if ew == 0 or ew == 255 or not (base <= ew <= base + 15):
            assert h == 0
        else:
            assert h == ((w >> 15) << 7) | ((ew - base) << 3) | ((w & 0x7F) >> 4)


def test_exhaustive_roundtrip_every_bf16_pattern(oracle):
    """All 65536 BF16 patterns (zeros, denormals, Inf, NaN payloads included)
    survive encode -> decode bit for bit."""
    W = synth.all_patterns(rows=64, seed=0)
    st, t = oracle.encode(W)
    assert st == oracle.OK
    st, D = oracle.decode(t)
    assert st == oracle.OK
    assert np.array_equal(D, W)
    check_invariants(oracle, W, t)
    st, nm = oracle.verify(W, t)
    assert st == oracle.OK and nm == 0


def test_roundtrip_single_window_rows(oracle):
    """Rows whose weights all lie in one 16-binade window need no escapes."""
    rng = np.random.default_rng(3)
    rows = []
    for n in range(40):
        b = int(rng.integers(1, 240))
        e = rng.integers(b, b + 16, size=333)
        s = rng.integers(0, 2, size=333)
        m = rng.integers(0, 128, size=333)
        rows.append(((s << 15) | (e << 7) | m).astype(np.uint16))
    W = np.stack(rows)
    st, t = oracle.encode(W)
    assert st == oracle.OK and t.n_esc == 0
    assert np.array_equal(oracle.decode(t)[1], W)
    check_invariants(oracle, W, t)


def test_roundtrip_dense_and_adversarial(oracle):
    for W in (synth.dense_weights(77, 300, seed=2), synth.adversarial_weights(130, 257, seed=4)):
        st, t = oracle.encode(W)
        assert st == oracle.OK
        assert np.array_equal(oracle.decode(t)[1], W)
        check_invariants(oracle, W, t)


def test_capacity_path_keeps_planes(oracle):
    W = synth.dense_weights(64, 512, seed=9)
    st, full = oracle.encode(W)
    assert st == oracle.OK and full.n_esc > 4
    cap = full.n_esc // 2
    st, part = oracle.encode(W, esc_cap=cap)
    assert st == oracle.ERR_CAPACITY and part.n_esc == full.n_esc
    for name in ("hi", "lo", "base", "esc_ptr"):
        assert np.array_equal(getattr(part, name), getattr(full, name))
    assert np.array_equal(part.esc[:cap], full.esc[:cap])


def test_bits_per_weight_gaussian_matches_pages(oracle):
    """Gaussian rows with a log-normal channel scale land in the pages'
    12.01-12.02 bits/weight regime."""
    with open(os.path.join(GOLDEN, "paper_figures.json")) as f:
        fig = json.load(f)
    W = synth.dense_weights(1024, 5120, seed=21, zero_frac=0.0, outlier_frac=0.0)
    st, t = oracle.encode(W)
    assert st == oracle.OK
    bpw = t.bits_per_weight()
    assert fig["bits_per_weight_low"] - 0.005 <= bpw <= fig["bits_per_weight_high"], bpw
    # the closed form of the accounting: 12 bits of planes, 8 bits of base per
    # row, a 32-bit offset per 16 x 256 group (+1), 32 bits per escape
    groups = 1024 // 16 * 5120 // 256
    assert bpw == pytest.approx(12.0 + 8 / 5120 + 32 * (groups + 1) / (1024 * 5120) + 32 * t.n_esc / (1024 * 5120))
    # escapes of a Gaussian row fall below the 16-binade window: ~6e-5
    assert 1e-5 < t.n_esc / W.size < 2e-4


def test_window_concentration_ratio_matches_pages(oracle):
    """The pages' 44.67 GB -> 33.58 GB ratio is ~12.03/16; the accounting of a
    Gaussian-like synthetic layer gives a size ratio within 0.002 of it."""
    with open(os.path.join(GOLDEN, "paper_figures.json")) as f:
        fig = json.load(f)
    W = synth.dense_weights(512, 5120, seed=22, zero_frac=0.0, outlier_frac=0.0)
    st, t = oracle.encode(W)
    ratio = t.bits_per_weight() / 16.0
    assert abs(ratio - fig["converted_layers_gb_after"] / fig["converted_layers_gb_before"]) < 0.002


def test_verify_counts_planted_corruption(oracle):
    """Corruption planted in a host copy gives the count the format implies."""
    W = synth.dense_weights(48, 320, seed=13)
    st, t = oracle.encode(W)
    Kp = oracle.cols_padded(320)
    esc = escaped_mask(W, t.base)
    rng = np.random.default_rng(0)
    # (1) a hi bit of an in-window weight: exactly one mismatch
    n, k = next((int(a), int(b)) for a, b in zip(rng.integers(0, 48, 999), rng.integers(0, 320, 999))
                if not esc[a, b])
    c = t.copy()
    c.hi[oracle.hi_offset(n, k, Kp)] ^= 0x10
    assert oracle.verify(W, c) == (oracle.ERR_MISMATCH, 1)
    # (2) the same bit under an escaped slot: hidden by the escape
    n2, k2 = map(int, np.argwhere(esc)[0])
    c = t.copy()
    c.hi[oracle.hi_offset(n2, k2, Kp)] ^= 0x10
    assert oracle.verify(W, c) == (oracle.OK, 0)
    # (3) a lo nibble bit: one mismatch
    c = t.copy()
    b, s = oracle.lo_position(n, k, Kp)
    c.lo[b] ^= (1 << s)
    assert oracle.verify(W, c) == (oracle.ERR_MISMATCH, 1)
    # (4) a base: every non-escaped weight of the row
    c = t.copy()
    c.base[5] ^= 1
    assert oracle.verify(W, c) == (oracle.ERR_MISMATCH, 320 - int(esc[5].sum()))
    # (5) an escape value: one mismatch
    c = t.copy()
    c.esc[3] ^= 0x0100
    assert oracle.verify(W, c) == (oracle.ERR_MISMATCH, 1)
    # (6) an escape key moved to another in-window weight of the same group:
    # two mismatches (the old slot loses its value, the new one gets it)
    c = t.copy()
    e = int(np.nonzero(np.diff(t.esc_ptr) >= 1)[0][0])
    first = int(t.esc_ptr[e])
    last = int(t.esc_ptr[e + 1]) - 1
    n0, k0 = t.position(last)
    k1 = next(kk for kk in range(k0 + 1, min(320, (k0 // 256 + 1) * 256)) if not esc[n0, kk]) \
        if any(not esc[n0, kk] for kk in range(k0 + 1, min(320, (k0 // 256 + 1) * 256))) else None
    if k1 is not None:
        c.esc[last] = (oracle.key(n0, k1) << 16) | (int(c.esc[last]) & 0xFFFF)
        assert oracle.verify(W, c) == (oracle.ERR_MISMATCH, 2)
    # (7) keys out of order inside a group: malformed
    c = t.copy()
    g = next(i for i in range(t.esc_ptr.size - 1) if t.esc_ptr[i + 1] - t.esc_ptr[i] >= 2)
    i = t.esc_ptr[g]
    c.esc[i], c.esc[i + 1] = c.esc[i + 1], c.esc[i]
    assert oracle.verify(W, c) == (oracle.ERR_CORRUPT, -1)
    # (8) a key naming a column past K: malformed
    c = t.copy()
    last_group = t.esc_ptr.size - 2  # group 1 of the last stripe covers columns 256..319
    c2 = t.copy()
    c2.esc_ptr[:] = t.esc_ptr
    if t.esc_ptr[last_group + 1] > t.esc_ptr[last_group]:
        j = int(t.esc_ptr[last_group + 1]) - 1
        key = (1 << 10) | (int(t.esc[j] >> 16) & 0x3C0) | 0x3F  # column 256+64+63 >= 320
        c2.esc[j] = (key << 16) | (int(t.esc[j]) & 0xFFFF)
        assert oracle.verify(W, c2) == (oracle.ERR_CORRUPT, -1)
