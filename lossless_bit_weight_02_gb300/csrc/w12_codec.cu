// W12 codec kernels: encode (window search; pack with the escape offsets),
// decode, load-time verify and escape-list structure check.
//
// All of them are HBM-bound integer work (SpecPilot, arXiv 2611.02501,
// section 4.1: conversion to W12 and the bit-for-bit check of every decoded
// tensor at load time).  Work is organised around the 16-row x 256-column
// group, the unit the escape list is indexed by.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

// Eight consecutive weights of a row as four words (weight 2i in the low
// half of word i); columns at or past K read as `fill`.
__device__ __forceinline__ uint4 load8w(const uint16_t *row, bool vec, int64_t k, int64_t K, uint32_t fill) {
    if (vec && k + 8 <= K) return __ldg(reinterpret_cast<const uint4 *>(row + k));
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a = (k + 2 * j < K) ? (uint32_t)row[k + 2 * j] : fill;
        const uint32_t b = (k + 2 * j + 1 < K) ? (uint32_t)row[k + 2 * j + 1] : fill;
        w[j] = a | (b << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The window test and the record field for two weights at once.  Per 16-bit
// half, window_word gives h = (w & 0x7FFF) + 0x8000 - (base << 7), that is
// 0x8000 + f with f = (w & 0x7FFF) - (base << 7) the record's offset-and-
// mantissa field (e-base)<<7 | m.  For any base byte h stays in
// [0x80, 0xFFFF], so no borrow or carry crosses the halves.  The weight lies
// in the window [base, base+15] exactly when 0 <= f <= 0x7FF, i.e. when
// h & 0xF800 == 0x8000: escape_bits is nonzero in the half of every weight
// outside its window (e = 0 and e = 255 included, since base is in [1, 239]).
__device__ __forceinline__ uint32_t window_c2(uint32_t b) { return 0x80008000u - b * 0x00800080u; }
__device__ __forceinline__ uint32_t window_word(uint32_t x, uint32_t c2) { return (x & 0x7FFF7FFFu) + c2; }
__device__ __forceinline__ uint32_t escape_bits(uint32_t d) { return (d & 0xF800F800u) ^ 0x80008000u; }

// ---------------------------------------------------------------------------
// a1: the window search, one of two kernels by row length.  Both build the
// exact histogram of the row's exponent field and take the window of 16
// consecutive exponents holding the most counted weights (exponents 0 and 255
// are always escapes and not counted; ties go to the largest base).  The grid
// also sets esc_ptr[0..P] to -1 ("not yet") for the pack kernel's look-back.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void red_add_shared(uint32_t a, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// The window base from a warp's counts, lane j holding h[i] = the count of
// exponent 8j + i (0 for exponents 0 and 255).
__device__ __forceinline__ int window_base(const uint32_t h[8], int lane) {
    // c[i] = number of counted weights with exponent <= 8*lane + i
    uint32_t c[8], run = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        run += h[i];
        c[i] = run;
    }
    uint32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - run;
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] += excl;
    // window b = 8*lane + i holds c(b+15) - c(b-1) weights: c(b+15) is lane
    // lane+1's c[7] for i = 0 and lane lane+2's c[i-1] otherwise
    uint32_t up[7];
#pragma unroll
    for (int i = 0; i < 7; ++i) up[i] = __shfl_down_sync(kFull, c[i], 2);
    const uint32_t next7 = __shfl_down_sync(kFull, c[7], 1);
    int best = -1, best_b = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int b = 8 * lane + i;
        const int cnt = (int)((i == 0 ? next7 : up[i - 1]) - (i == 0 ? excl : c[i - 1]));
        if (b >= 1 && b <= 239 && cnt >= best) {  // b ascending: ties go to the larger base
            best = cnt;
            best_b = b;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const int ob = __shfl_xor_sync(kFull, best, o);
        const int obb = __shfl_xor_sync(kFull, best_b, o);
        if (ob > best || (ob == best && obb > best_b)) {
            best = ob;
            best_b = obb;
        }
    }
    return best_b;
}

constexpr int64_t kLongRow = 8192;  // columns: longer rows take the 4-warp kernel

// Block n of an n_blocks grid sets its share of esc_ptr[0..P] to -1.
__device__ __forceinline__ void mark_not_ready(int32_t *esc_ptr, int64_t P, int64_t n, int64_t n_blocks, int t,
                                               int nt) {
    for (int64_t i = n + n_blocks * t; i <= P; i += n_blocks * nt) esc_ptr[i] = -1;
}

// Rows of at most kLongRow columns: one warp (and block) per row, 24 rows in
// flight per SM.  The histogram lives in shared memory as 8-bit counters
// private to each lane: exponent e of lane L is byte e/64 of the word at
// (e%64)*128 + 4L.  A lane only ever touches its own bank (one shared
// histogram took the lanes that hit the same exponent one after another), and
// the low weight of a word x finds its counter word as (x & 0x1F80) | 4L,
// exponent bits 0..5 already in place; the add is a shared-memory reduction
// (a plain load, add and store measured 14% slower).  Every exponent is
// counted, 0 and 255 included; those two bins are dropped before the window
// search.  A lane adds 8 weights per 256-column step, so the counters are
// folded into per-lane totals every 28 steps, before they can pass 255.
// ---------------------------------------------------------------------------
constexpr int kFoldSteps = 28;  // 28 * 8 = 224 < 256 adds per counter between folds

// 1 << 8 * (c & 3): byte c & 3 of the result is 1.  prmt's backward
// 4-extract mode reads the selector's two low bits only and puts source byte
// 0 (here the 1) at result byte c & 3, the others from source bytes 1..7 (0).
__device__ __forceinline__ uint32_t byte_one(uint32_t c) {
    uint32_t d;
    asm("prmt.b32.b4e %0, %1, %2, %3;" : "=r"(d) : "r"(1u), "r"(0u), "r"(c));
    return d;
}

// hl = the shared address of the counters + 4 * lane.  Exponent bits 6 and 7
// of the low weight are bits 13 and 14 of x (bit 15, the sign, lands in the
// selector's bit 2, which the extract ignores); of the high weight, 29 and 30.
__device__ __forceinline__ void count_word(uint32_t hl, uint32_t x) {
    red_add_shared(hl + (x & 0x1F80u), byte_one(x >> 13));
    const uint32_t h = x >> 16;
    red_add_shared(hl + (h & 0x1F80u), byte_one(h >> 13));
}

// Lane j adds counter words j and j+32 of all 32 copies (reading copy
// (i + j) % 32 at step i: distinct banks) into tot[m] = count of exponent
// j + 32m, and optionally clears what it read.
__device__ __forceinline__ void fold_counts(uint32_t *h, int lane, bool clear, uint32_t tot[8]) {
    __syncwarp();
    uint32_t a0 = 0, b0 = 0, a1 = 0, b1 = 0;  // two 16-bit sums each (at most 32 * 224)
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
        const int c = (i + lane) & 31;
        const uint32_t x0 = h[32 * lane + c], x1 = h[32 * (lane + 32) + c];
        if (clear) {
            h[32 * lane + c] = 0u;
            h[32 * (lane + 32) + c] = 0u;
        }
        a0 += x0 & 0x00FF00FFu;         // exponents j (low) and j + 128 (high)
        b0 += (x0 >> 8) & 0x00FF00FFu;  // j + 64, j + 192
        a1 += x1 & 0x00FF00FFu;         // j + 32, j + 160
        b1 += (x1 >> 8) & 0x00FF00FFu;  // j + 96, j + 224
    }
    tot[0] += a0 & 0xFFFFu;
    tot[1] += a1 & 0xFFFFu;
    tot[2] += b0 & 0xFFFFu;
    tot[3] += b1 & 0xFFFFu;
    tot[4] += a0 >> 16;
    tot[5] += a1 >> 16;
    tot[6] += b0 >> 16;
    tot[7] += b1 >> 16;
    __syncwarp();
}

// Calls f(s, x) for the steps s = 0 .. full-1 of a row, x = this lane's 8
// weights of step s (p[32 * s]), with four steps in flight per warp (24
// warps per SM then keep ~48 KB of loads in flight, enough to cover HBM
// latency).
template <class F>
__device__ __forceinline__ void for_full_steps(const uint4 *__restrict__ p, int full, F &&f) {
    int s = 0;
    if (full >= 8) {
        uint4 n0 = __ldg(p), n1 = __ldg(p + 32), n2 = __ldg(p + 64), n3 = __ldg(p + 96);
        for (; s + 8 <= full; s += 4) {
            uint4 x = n0;
            n0 = __ldg(p + 32 * (s + 4));
            f(s, x);
            x = n1;
            n1 = __ldg(p + 32 * (s + 5));
            f(s + 1, x);
            x = n2;
            n2 = __ldg(p + 32 * (s + 6));
            f(s + 2, x);
            x = n3;
            n3 = __ldg(p + 32 * (s + 7));
            f(s + 3, x);
        }
        f(s, n0);
        f(s + 1, n1);
        f(s + 2, n2);
        f(s + 3, n3);
        s += 4;
    }
    for (; s < full; ++s) f(s, __ldg(p + 32 * s));
}

__global__ __launch_bounds__(32) void k_window_warp(const uint16_t *__restrict__ W, int64_t ldw, int64_t N, int64_t K,
                                                   uint8_t *__restrict__ base, int32_t *__restrict__ esc_ptr,
                                                   int64_t P) {
    __shared__ __align__(16) uint32_t hist[64 * 32];  // [e % 64][lane], byte e / 64
    const int lane = threadIdx.x;
    const int64_t n = blockIdx.x;
    const uint32_t hl = (uint32_t)__cvta_generic_to_shared(hist) + (uint32_t)lane * 4u;
#pragma unroll 8
    for (int w = 0; w < 64; ++w) hist[32 * w + lane] = 0u;
    __syncwarp();
    const uint16_t *row = W + n * ldw;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int G = (int)groups_of(K);                  // steps of 256 columns (G < 2^24: checked on the host)
    const int full = vec ? (int)(K >> 8) : 0;        // steps whose 8 columns are in range for every lane
    const uint4 *p = reinterpret_cast<const uint4 *>(row) + lane;  // step s: p[32 * s]
    uint32_t tot[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int since = 0;
    auto count_step = [&](int s, const uint4 &x) {
        count_word(hl, x.x);
        count_word(hl, x.y);
        count_word(hl, x.z);
        count_word(hl, x.w);
        if (++since == kFoldSteps && s + 1 < G) {
            fold_counts(hist, lane, true, tot);
            since = 0;
        }
    };
    for_full_steps(p, full, count_step);
    // the partial step (or every step of an unaligned row): past K reads as
    // exponent 0, dropped
    for (int s = full; s < G; ++s) count_step(s, load8w(row, vec, (int64_t)s * 256 + lane * 8, K, 0u));
    fold_counts(hist, lane, false, tot);
    if (lane == 0) tot[0] = 0;    // exponent 0: zeros and subnormals are escapes
    if (lane == 31) tot[7] = 0;   // exponent 255: infinities and NaNs too
    // regroup through shared memory: lane j then holds exponents 8j..8j+7
#pragma unroll
    for (int m = 0; m < 8; ++m) hist[lane + 32 * m] = tot[m];
    __syncwarp();
    const uint4 t0 = reinterpret_cast<const uint4 *>(hist)[2 * lane], t1 = reinterpret_cast<const uint4 *>(hist)[2 * lane + 1];
    const uint32_t h[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
    const int best_b = window_base(h, lane);
    if (lane == 0) base[n] = (uint8_t)best_b;
    mark_not_ready(esc_ptr, P, n, N, lane, 32);
}

// Longer rows: one block of 4 warps per row, warp w taking the row's
// 256-column steps w, w+4, ...  A row's fixed costs (clearing and summing the
// table, the search) are spread over more columns, and a row's steps are
// spread over more warps.
//
// The histogram is a shared-memory table of 32-bit counters with one column
// per lane index: exponent e, lane L at byte 128*e + 4L, i.e. the counter of
// the low weight of a word x sits at (x & 0x7F80) | 4L.  So a weight costs one
// mask and one shared-memory reduction of a constant 1: no increment to build
// and no lane ever collides with another lane of its warp (one counter per
// exponent took the lanes that hit the same exponent one after another).
// Lanes of the same index in the block's four warps share a column; their
// reductions are separate instructions and need no ordering.  Every exponent
// is counted, 0 and 255 included; those two bins are dropped before the
// window search.
// ---------------------------------------------------------------------------
constexpr int kRowWarps = 4;

// hl = shared address of the table + 4 * lane
__device__ __forceinline__ void count_word32(uint32_t hl, uint32_t x) {
    red_add_shared(hl + (x & 0x7F80u), 1u);
    red_add_shared(hl + ((x >> 16) & 0x7F80u), 1u);
}

// Calls f(s, x) for this warp's steps s = w, w + 4, ... below `full` of a
// row, x = this lane's 8 weights of step s (p[32 * s]), with four of the
// warp's steps in flight.
template <class F>
__device__ __forceinline__ void for_warp_steps(const uint4 *__restrict__ p, int w, int full, F &&f) {
    int s = w;
    if (s + 12 < full) {
        uint4 n0 = __ldg(p + 32 * s), n1 = __ldg(p + 32 * (s + 4));
        uint4 n2 = __ldg(p + 32 * (s + 8)), n3 = __ldg(p + 32 * (s + 12));
        for (; s + 28 < full; s += 16) {
            uint4 x = n0;
            n0 = __ldg(p + 32 * (s + 16));
            f(s, x);
            x = n1;
            n1 = __ldg(p + 32 * (s + 20));
            f(s + 4, x);
            x = n2;
            n2 = __ldg(p + 32 * (s + 24));
            f(s + 8, x);
            x = n3;
            n3 = __ldg(p + 32 * (s + 28));
            f(s + 12, x);
        }
        f(s, n0);
        f(s + 4, n1);
        f(s + 8, n2);
        f(s + 12, n3);
        s += 16;
    }
    for (; s < full; s += 4) f(s, __ldg(p + 32 * s));
}

__global__ __launch_bounds__(kRowWarps * 32) void k_window_block(const uint16_t *__restrict__ W, int64_t ldw,
                                                               int64_t N, int64_t K, uint8_t *__restrict__ base,
                                                               int32_t *__restrict__ esc_ptr, int64_t P) {
    __shared__ __align__(16) uint32_t hist[256 * 32];  // [exponent][lane]
    __shared__ uint32_t tot[256];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = blockIdx.x;
#pragma unroll
    for (int i = 0; i < 16; ++i) reinterpret_cast<uint4 *>(hist)[i * 128 + tid] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const uint16_t *row = W + n * ldw;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int G = (int)groups_of(K);            // 256-column steps (K < 2^31: checked on the host)
    const int full = vec ? (int)(K >> 8) : 0;  // steps whose 8 columns are in range for every lane
    const uint4 *p = reinterpret_cast<const uint4 *>(row) + lane;  // step s: p[32 * s]
    const uint32_t hl = (uint32_t)__cvta_generic_to_shared(hist) + (uint32_t)lane * 4u;
    auto count_step = [&](int, const uint4 &x) {
        count_word32(hl, x.x);
        count_word32(hl, x.y);
        count_word32(hl, x.z);
        count_word32(hl, x.w);
    };
    for_warp_steps(p, warp, full, count_step);
    // the partial step (or every step of an unaligned row): past K reads as
    // exponent 0, dropped
    for (int s = (full > warp ? full + ((warp - full) & 3) : warp); s < G; s += 4)
        count_step(s, load8w(row, vec, (int64_t)s * 256 + lane * 8, K, 0u));
    __syncthreads();
    // thread t sums exponents 2t and 2t+1 over the 32 lane columns (128-byte
    // rows read as eight 16-byte pieces, rotated by lane: conflict-free)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = 2 * tid + h;
        const uint4 *r = reinterpret_cast<const uint4 *>(hist + 32 * e);
        uint32_t s = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = r[(c + lane) & 7];
            s += v.x + v.y + v.z + v.w;
        }
        tot[e] = (e == 0 || e == 255) ? 0u : s;  // exponents 0 and 255 are always escapes
    }
    __syncthreads();
    if (warp == 0) {
        const uint4 t0 = reinterpret_cast<const uint4 *>(tot)[2 * lane], t1 = reinterpret_cast<const uint4 *>(tot)[2 * lane + 1];
        const uint32_t h[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        const int b = window_base(h, lane);
        if (lane == 0) base[n] = (uint8_t)b;
    }
    mark_not_ready(esc_ptr, P, n, N, tid, kRowWarps * 32);
}

// ---------------------------------------------------------------------------
// a2 + a3: pack, with the escape offsets found on the way (k_pack, one
// cooperative launch of resident blocks).
//  1. Units (16-row stripe t, 256-column group g) are handed out one at a
//     time from a counter in esc_ptr[0], so fast SMs take more, last unit
//     first: the window kernel read the last rows last, and part of them is
//     still in L2.  A warp packs
//     unit u into tiles 4u .. 4u+3 of the planes (4 KB of hi bytes, 2 KB of lo
//     bytes, contiguous).  Lane (r = lane/4, q = lane%4) takes columns
//     16q..16q+15 of rows r and r+8 of each tile: exactly one 16-byte slot of
//     the hi tile per row (the hi tile is row-major, byte 64*row + column)
//     and one 16-byte slot of the lo tile, so every store is a coalesced
//     512-byte warp store.  The whole 8 KB unit is loaded before it is
//     packed, and the block keeps little shared memory, so L1 can hold the
//     loads of 16 warps in flight.  The unit's escapes, in (tile, row, column)
//     order (rows r in lane order, then rows r+8, per tile, by a warp scan of
//     per-lane counts), are staged in the warp's shared memory, and its
//     esc_ptr slot gets its count as a code (below).
//  2. A grid barrier (arrivals counted on the same counter).
//  3. Block b scans the counts of units [b*SEG, (b+1)*SEG): it publishes the
//     segment's total in the slot of its last unit (-2 - total), reads the
//     slots of the segments before it until it meets an inclusive total
//     (decoupled look-back, all threads reading at once), publishes its own
//     inclusive total and writes the offsets of its units.
//  4. A second grid barrier; then every warp copies its staged escapes to
//     their offsets.  A unit whose escapes did not fit the staging area is
//     re-derived from W by its scan block in step 3.
// Slot codes while the kernel runs: -1 not yet (set by the window kernel), at
// most kCountCode0 a unit's count from step 1, -2 .. kAggMin a segment total,
// >= 0 an inclusive total, kEncTimeout / kEncOverflow an inclusive total that
// carries an error.
// ---------------------------------------------------------------------------
constexpr int kPackWarps = 4;     // 151 registers (a whole unit in flight): three 4-warp blocks per SM
constexpr int kPackStage = 640;   // escape words a warp holds until the offsets are known
constexpr int kPackList = 128;    // units a warp holds escapes for
constexpr int kPackRedo = 256;    // unstaged units a scan block remembers (more: it redoes its segment)
constexpr int32_t kEncNotReady = -1;
constexpr int32_t kEncTimeout = INT32_MIN;  // inclusive totals that carry an error
constexpr int32_t kEncOverflow = INT32_MIN + 1;
constexpr int32_t kAggMin = -(1 << 30) + 1;        // segment totals: -2 - total, total <= 2^30 - 3
constexpr int32_t kCountCode0 = -(1 << 30) - 1;    // a unit's count c: kCountCode0 - c (- kUnstaged)
constexpr int32_t kUnstaged = 1 << 20;             // ... if its escapes are not in the staging area
constexpr uint32_t kEncPollLimit = 1u << 21;       // polls of a wait (backoff to 256 ns): about 2 s

// Sixteen weights of a row (columns k..k+15) as eight words; columns past K
// read as `fill`.
__device__ __forceinline__ void load16w(const uint16_t *row, bool vec, int64_t k, int64_t K, uint32_t fill,
                                        uint32_t x[8]) {
    const uint4 a = load8w(row, vec, k, K, fill), b = load8w(row, vec, k + 8, K, fill);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Hi bytes of a word's two weights (bytes 0 and 2; 1 and 3 are don't-care):
// sign << 7 | f >> 4, i.e. the 12-bit record s<<11 | f shifted right by 4.
__device__ __forceinline__ uint32_t hi_pair(uint32_t d, uint32_t x) {
    return ((d >> 4) & 0x007F007Fu) | ((x >> 8) & 0xFF80FF80u);
}

// The slot's 16 hi bytes, column c at byte c.
__device__ __forceinline__ uint4 hi_slot(const uint32_t d[8], const uint32_t x[8]) {
    return make_uint4(prmt(hi_pair(d[0], x[0]), hi_pair(d[1], x[1]), 0x6420),
                      prmt(hi_pair(d[2], x[2]), hi_pair(d[3], x[3]), 0x6420),
                      prmt(hi_pair(d[4], x[4]), hi_pair(d[5], x[5]), 0x6420),
                      prmt(hi_pair(d[6], x[6]), hi_pair(d[7], x[7]), 0x6420));
}

// A lo word of eight columns c0..c0+7: byte u = lo(c0+u) << 4 | lo(c0+u+4),
// the record's low nibble being f & 0xF.
__device__ __forceinline__ uint32_t lo_word(uint32_t d0, uint32_t d1, uint32_t d2, uint32_t d3) {
    const uint32_t a = prmt(d0, d1, 0x6420), b = prmt(d2, d3, 0x6420);
    return ((a << 4) & 0xF0F0F0F0u) | (b & 0x0F0F0F0Fu);
}

// The escape mask of a lane's 16 columns of one tile row: bit c is set when
// column 16q + c is an escape.
__device__ __forceinline__ uint32_t escape_mask(const uint32_t d[8]) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t e = escape_bits(d[i]);
        m |= (uint32_t)((e & 0xFFFFu) != 0u) << (2 * i) | (uint32_t)((e >> 16) != 0u) << (2 * i + 1);
    }
    return m;
}

// Writes the escapes of mask m (keys key0 + c, values from x) to esc[pos...]
// below esc_lim and turns their records into 0 (d = 0x8000, sign cleared).
__device__ __forceinline__ void put_escapes(uint32_t m, uint32_t d[8], uint32_t x[8], uint32_t key0, int64_t pos,
                                            uint64_t esc_lim, uint32_t *__restrict__ esc) {
    for (uint32_t mm = m; mm; mm &= mm - 1u, ++pos) {
        const int c = __ffs(mm) - 1;
        // the word of column c, picked by selects (no indexed array access)
        const uint32_t w01 = (c & 2) ? x[1] : x[0], w23 = (c & 2) ? x[3] : x[2];
        const uint32_t w45 = (c & 2) ? x[5] : x[4], w67 = (c & 2) ? x[7] : x[6];
        const uint32_t w03 = (c & 4) ? w23 : w01, w47 = (c & 4) ? w67 : w45;
        const uint32_t w = (c & 8) ? w47 : w03;
        const uint32_t v = (c & 1) ? (w >> 16) : (w & 0xFFFFu);
        if ((uint64_t)pos < esc_lim) esc[pos] = ((key0 + (uint32_t)c) << 16) | v;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t z = ((m >> (2 * i)) & 1u ? 0x0000FFFFu : 0u) | ((m >> (2 * i + 1)) & 1u ? 0xFFFF0000u : 0u);
        d[i] = (d[i] & ~z) | (0x80008000u & z);
        x[i] &= ~(z & 0x80008000u);
    }
}

// The escapes among this lane's columns 16q..16q+15 of tile rows r (d0, x0)
// and r+8 (d1, x1) (a warp-wide call): written after the `p` entries the unit
// already holds, in (row, column) order, i.e. row r of every lane in lane
// order, then row r+8.  One warp scan ranks both rows (a 16-bit count each);
// only the lanes that hold an escape (a few per tile) walk their set bits.
__device__ __forceinline__ void pack_escapes(uint32_t d0[8], uint32_t x0[8], bool any0, uint32_t d1[8],
                                             uint32_t x1[8], bool any1, int c4, int r, int q, int lane, int64_t &p,
                                             uint64_t esc_lim, uint32_t *__restrict__ esc) {
    const uint32_t m0 = any0 ? escape_mask(d0) : 0u, m1 = any1 ? escape_mask(d1) : 0u;
    const uint32_t n0 = __popc(m0), n1 = __popc(m1);
    uint32_t incl = n0 | (n1 << 16);  // at most 32 * 16 per half: no carry
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t tot = __shfl_sync(kFull, incl, 31);
    const int64_t pos0 = p + (int64_t)((incl & 0xFFFFu) - n0);
    const int64_t pos1 = p + (int64_t)(tot & 0xFFFFu) + (int64_t)((incl >> 16) - n1);
    p += (int64_t)(tot & 0xFFFFu) + (int64_t)(tot >> 16);
    const uint32_t key = (uint32_t)(c4 << 10) | (uint32_t)(r << 6) | (uint32_t)(16 * q);
    if (m0) put_escapes(m0, d0, x0, key, pos0, esc_lim, esc);
    if (m1) put_escapes(m1, d1, x1, key + (8u << 6), pos1, esc_lim, esc);
}

// Packs unit u (a warp-wide call) into its planes and writes its escapes to
// escd[p...] below lim, p advancing by their count.
__device__ __forceinline__ void pack_unit(const uint16_t *__restrict__ W, int64_t ldw, int64_t N, int64_t K,
                                          const uint8_t *__restrict__ base, uint8_t *__restrict__ hi,
                                          uint8_t *__restrict__ lo, int64_t u, int64_t G, int lane, int64_t &p,
                                          uint64_t lim, uint32_t *escd) {
    const int64_t t = u / G, g = u - t * G;
    const int r = lane >> 2, q = lane & 3;
    const int64_t nA = t * 16 + r, nB = nA + 8;
    // a padding row (n >= N) reads nothing: base 0 and fill 0 give record 0
    const bool okA = nA < N, okB = nB < N;
    const uint32_t bA = okA ? base[nA] : 0u, bB = okB ? base[nB] : 0u;
    const uint32_t c2A = window_c2(bA), c2B = window_c2(bB), fA = bA << 7, fB = bB << 7;
    const uint16_t *rowA = W + (okA ? nA : 0) * ldw, *rowB = W + (okB ? nB : 0) * ldw;
    const int64_t KA = okA ? K : 0, KB = okB ? K : 0;
    const bool vecA = (reinterpret_cast<uintptr_t>(rowA) & 15) == 0, vecB = (reinterpret_cast<uintptr_t>(rowB) & 15) == 0;
    uint4 *hu = reinterpret_cast<uint4 *>(hi + u * 4096);
    uint4 *lu = reinterpret_cast<uint4 *>(lo + u * 2048);
    // a whole unit in range and aligned is loaded up front (8 KB per warp in
    // flight) with plain 16-byte loads; a ragged or padding edge, or an
    // unaligned row, takes bounds-checked loads per tile (warp-uniform choice)
    const bool fast = okB && vecA && vecB && (g + 1) * 256 <= K;
    uint4 A[8], B[8];
    if (fast) {
        const uint4 *pa = reinterpret_cast<const uint4 *>(rowA + g * 256 + 16 * q);
        const uint4 *pb = reinterpret_cast<const uint4 *>(rowB + g * 256 + 16 * q);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            A[j] = __ldg(pa + 8 * (j >> 1) + (j & 1));
            B[j] = __ldg(pb + 8 * (j >> 1) + (j & 1));
        }
    }
    // one tile per pass, not unrolled (the loop then fits the instruction
    // cache): the unit's registers move down by a tile after each pass
#pragma unroll 1
    for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t xa[8], xb[8];
        if (fast) {
            const uint4 u0 = A[0], u1 = A[1], v0 = B[0], v1 = B[1];
            xa[0] = u0.x, xa[1] = u0.y, xa[2] = u0.z, xa[3] = u0.w, xa[4] = u1.x, xa[5] = u1.y, xa[6] = u1.z, xa[7] = u1.w;
            xb[0] = v0.x, xb[1] = v0.y, xb[2] = v0.z, xb[3] = v0.w, xb[4] = v1.x, xb[5] = v1.y, xb[6] = v1.z, xb[7] = v1.w;
        } else {
            const int64_t k = g * 256 + c4 * 64 + 16 * q;
            load16w(rowA, vecA, k, KA, fA, xa);
            load16w(rowB, vecB, k, KB, fB, xb);
        }
        uint32_t da[8], db[8], ea = 0, eb = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            da[i] = window_word(xa[i], c2A);
            db[i] = window_word(xb[i], c2B);
            ea |= escape_bits(da[i]);
            eb |= escape_bits(db[i]);
        }
        if (__any_sync(kFull, (ea | eb) != 0u)) {
            pack_escapes(da, xa, ea != 0u, db, xb, eb != 0u, c4, r, q, lane, p, lim, escd);
        }
        hu[c4 * 64 + lane] = hi_slot(da, xa);
        hu[c4 * 64 + 32 + lane] = hi_slot(db, xb);
        lu[c4 * 32 + lane] = make_uint4(lo_word(da[0], da[1], da[2], da[3]), lo_word(da[4], da[5], da[6], da[7]),
                                        lo_word(db[0], db[1], db[2], db[3]), lo_word(db[4], db[5], db[6], db[7]));
        if (fast) {
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                A[j] = A[j + 2];
                B[j] = B[j + 2];
            }
        }
    }
}

__device__ __forceinline__ int32_t ld_status(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_status(int32_t *p, int32_t v) {
    asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The escape offset of segment k (a block-wide call): the sum of the totals
// of the segments before it, read from their status slots esc_ptr[(j+1)*SEG].
// The block reads up to 512 slots per round trip: every segment is scanned at
// once, so the nearest inclusive total can sit many segments back.  A
// negative result is an error code taken over from a segment before, or
// kEncTimeout if a segment before published nothing within the poll limit.
struct LookbackSmem {
    long long sum[kPackWarps];
    long long jmax[kPackWarps];
    int flags[kPackWarps];
};
__device__ __forceinline__ long long segment_offset(const int32_t *esc_ptr, int64_t k, int64_t SEG, LookbackSmem &sh) {
    constexpr int NT = kPackWarps * 32, R = 4, WIN = NT * R;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    long long E = 0;
    int64_t top = k - 1;  // the highest segment not yet summed
    uint32_t polls = 0;
    unsigned ns = 64;
    while (top >= 0) {
        int32_t v[R];
        int64_t jj[R];
        long long mine = -2;  // the highest of this thread's segments with an inclusive total
#pragma unroll
        for (int r = 0; r < R; ++r) {
            jj[r] = top - tid - (int64_t)NT * r;
            v[r] = jj[r] >= 0 ? ld_status(esc_ptr + (jj[r] + 1) * SEG) : kEncNotReady;
            if (jj[r] >= 0 && (v[r] >= 0 || v[r] <= kEncOverflow) && jj[r] > mine) mine = jj[r];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const long long y = __shfl_xor_sync(kFull, mine, o);
            mine = y > mine ? y : mine;
        }
        if (lane == 0) sh.jmax[warp] = mine;
        __syncthreads();
        long long J = sh.jmax[0];
#pragma unroll
        for (int w = 1; w < kPackWarps; ++w) J = sh.jmax[w] > J ? sh.jmax[w] : J;
        if (J == -2 && top - WIN + 1 <= 0) J = -1;  // segment 0 starts at offset 0
        // the segments above J must all have published a total
        long long a = 0;
        int notready = 0, poison = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (jj[r] < 0 || jj[r] < J) continue;
            if (jj[r] == J) {
                if (v[r] < 0) poison = v[r];
                else a += v[r];
            } else if (v[r] == kEncNotReady || v[r] < kAggMin) {  // no total yet
                notready = 1;
            } else {
                a += (long long)(-2 - v[r]);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            a += __shfl_xor_sync(kFull, a, o);
            notready |= __shfl_xor_sync(kFull, notready, o);
            poison |= __shfl_xor_sync(kFull, poison, o);
        }
        __syncthreads();  // every thread has read jmax
        if (lane == 0) {
            sh.sum[warp] = a;
            sh.flags[warp] = notready;
            sh.jmax[warp] = poison;
        }
        __syncthreads();
        a = 0;
        notready = 0;
        poison = 0;
#pragma unroll
        for (int w = 0; w < kPackWarps; ++w) {
            a += sh.sum[w];
            notready |= sh.flags[w];
            poison |= (int)sh.jmax[w];
        }
        __syncthreads();  // before the next round writes the scratch
        if (notready) {
            if (++polls > kEncPollLimit) return kEncTimeout;
            __nanosleep(ns);
            if (ns < 256) ns *= 2;
            continue;
        }
        if (poison) return poison;  // an error code (both are negative, ORs of one code)
        E += a;
        if (J >= -1) break;
        top -= WIN;
    }
    return E > 0x7FFFFFFFLL ? (long long)kEncOverflow : E;
}

// Re-derives the escapes of unit u into esc[p...] below lim (a warp-wide
// call, the slow path of a warp whose escapes outgrew its staging area).
__device__ __noinline__ void unit_escapes(const uint16_t *__restrict__ W, int64_t ldw, int64_t N, int64_t K,
                                          const uint8_t *__restrict__ base, int64_t u, int64_t G, int64_t p,
                                          uint64_t lim, uint32_t *__restrict__ esc, int lane) {
    const int64_t t = u / G, g = u - t * G;
    const int r = lane >> 2, q = lane & 3;
    const int64_t nA = t * 16 + r, nB = nA + 8;
    const bool okA = nA < N, okB = nB < N;
    const uint32_t bA = okA ? base[nA] : 0u, bB = okB ? base[nB] : 0u;
    const uint32_t c2A = window_c2(bA), c2B = window_c2(bB), fA = bA << 7, fB = bB << 7;
    const uint16_t *rowA = W + (okA ? nA : 0) * ldw, *rowB = W + (okB ? nB : 0) * ldw;
    const int64_t KA = okA ? K : 0, KB = okB ? K : 0;
    const bool vecA = (reinterpret_cast<uintptr_t>(rowA) & 15) == 0, vecB = (reinterpret_cast<uintptr_t>(rowB) & 15) == 0;
    for (int c4 = 0; c4 < 4; ++c4) {
        const int64_t k = g * 256 + c4 * 64 + 16 * q;
        uint32_t xa[8], xb[8], da[8], db[8], ea = 0, eb = 0;
        load16w(rowA, vecA, k, KA, fA, xa);
        load16w(rowB, vecB, k, KB, fB, xb);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            da[i] = window_word(xa[i], c2A);
            db[i] = window_word(xb[i], c2B);
            ea |= escape_bits(da[i]);
            eb |= escape_bits(db[i]);
        }
        if (__any_sync(kFull, (ea | eb) != 0u)) {
            pack_escapes(da, xa, ea != 0u, db, xb, eb != 0u, c4, r, q, lane, p, lim, esc);
        }
    }
}

// Arrives at a grid barrier counted on *ctr and waits, within the poll
// limit, until it reads at least `target` (or 0: the counter was reset after
// the last barrier).  One thread per block.
__device__ __forceinline__ bool grid_barrier(int32_t *ctr, int64_t target) {
    __threadfence();
    atomicAdd(ctr, 1);
    unsigned ns = 32;
    for (uint32_t i = 0; i < kEncPollLimit; ++i) {
        const int32_t v = ld_status(ctr);
        if (v >= target || v == 0) {
            __threadfence();
            return true;
        }
        __nanosleep(ns);
        if (ns < 256) ns *= 2;
    }
    return false;
}

// The next unit for this warp: counter value + 1 (the counter starts at -1).
__device__ __forceinline__ int64_t next_unit(int32_t *ctr, int lane) {
    int v = 0;
    if (lane == 0) v = atomicAdd(ctr, 1);
    return (int64_t)__shfl_sync(kFull, v, 0) + 1;
}

__global__ __launch_bounds__(kPackWarps * 32, 3) void k_pack(const uint16_t *__restrict__ W, int64_t ldw, int64_t N,
                                                             int64_t K, const uint8_t *__restrict__ base,
                                                             int32_t *__restrict__ esc_ptr, uint8_t *__restrict__ hi,
                                                             uint8_t *__restrict__ lo, uint32_t *__restrict__ esc,
                                                             int64_t esc_cap, int64_t P, int64_t G,
                                                             int32_t *__restrict__ total, int test_stall) {
    __shared__ uint32_t stage[kPackWarps][kPackStage];
    __shared__ int32_t list_u[kPackWarps][kPackList];
    __shared__ int32_t list_c[kPackWarps][kPackList];
    __shared__ int32_t redo[kPackRedo];
    __shared__ int n_redo;
    __shared__ LookbackSmem lb;
    __shared__ int sync_ok;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NT = kPackWarps * 32;
    const int64_t B = gridDim.x;

    // 1. pack units as they are handed out
    int nl = 0;
    {
        int64_t p = 0;
        int64_t d = next_unit(esc_ptr, lane);
        while (d < P) {
            const int64_t u = P - 1 - d;
            // the next draw is in flight while this unit is packed
            int vn = 0;
            if (lane == 0) vn = atomicAdd(esc_ptr, 1);
            const int64_t p0 = p;
            pack_unit(W, ldw, N, K, base, hi, lo, u, G, lane, p, kPackStage, stage[warp]);
            const int c = (int)(p - p0);
            const bool staged = p <= kPackStage && nl < kPackList;
            if (staged) {
                if (lane == 0) {
                    list_u[warp][nl] = (int32_t)u;
                    list_c[warp][nl] = c;
                }
                ++nl;
            } else {
                p = p0;
            }
            if (lane == 0) esc_ptr[u + 1] = kCountCode0 - c - (staged ? 0 : kUnstaged);
            d = (int64_t)__shfl_sync(kFull, vn, 0) + 1;
        }
    }
    // 2. every count is in place: the counter has seen P + one failed draw
    // per warp and one arrival per block
    __syncthreads();
    if (tid == 0) {
        n_redo = 0;
        // the test hook: block 0 never arrives, so every block's wait runs out
        const bool arrive = !(test_stall && blockIdx.x == 0);
        sync_ok = arrive && grid_barrier(esc_ptr, P - 1 + (kPackWarps + 1) * B);
    }
    __syncthreads();
    // 3. scan segment b: units [s0, s1), status slot esc_ptr[s1]
    const int64_t SEG = (P + B - 1) / B, s0 = blockIdx.x * SEG, s1 = (s0 + SEG < P) ? s0 + SEG : P;
    if (s0 < s1) {
        // local inclusive totals replace the codes (all but the status slot,
        // whose code is read first), in tiles of NT
        long long run = 0;
        for (int64_t c0 = s0; c0 < s1; c0 += NT) {
            const int64_t u = c0 + tid;
            int32_t cnt = 0;
            if (u < s1) {
                const int32_t code = __ldcg(esc_ptr + u + 1);
                const int32_t x = kCountCode0 - code;
                cnt = x & (kUnstaged - 1);
                if (x & kUnstaged) {
                    const int i = atomicAdd(&n_redo, 1);
                    if (i < kPackRedo) redo[i] = (int32_t)(u - s0);
                }
            }
            int x = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) lb.sum[warp] = x;
            __syncthreads();
            long long before = run;
            for (int w = 0; w < warp; ++w) before += lb.sum[w];
            long long tile = 0;
            for (int w = 0; w < kPackWarps; ++w) tile += lb.sum[w];
            if (u < s1 && u + 1 != s1) {
                const long long v = before + x;
                esc_ptr[u + 1] = (int32_t)(v < 0x7FFFFFFFLL ? v : 0x7FFFFFFFLL);
            }
            run += tile;
            __syncthreads();
        }
        const long long agg = run;
        const bool big = agg > -2LL - kAggMin;
        if (tid == 0) st_status(esc_ptr + s1, big ? kEncOverflow : (int32_t)(-2 - agg));
        long long E = kEncTimeout;
        if (!sync_ok) {
            if (tid == 0) st_status(esc_ptr + s1, kEncTimeout);
        } else if (big) {
            E = kEncOverflow;
        } else {
            E = segment_offset(esc_ptr, blockIdx.x, SEG, lb);
            if (tid == 0) {
                const long long incl = E < 0 ? E : (E + agg > 0x7FFFFFFFLL ? (long long)kEncOverflow : E + agg);
                st_status(esc_ptr + s1, (int32_t)incl);
            }
        }
        for (int64_t u = s0 + tid; u + 1 < s1; u += NT) {
            const long long v = E + esc_ptr[u + 1];
            esc_ptr[u + 1] = (E < 0 || v > 0x7FFFFFFFLL) ? -1 : (int32_t)v;
        }
        __syncthreads();  // the segment's offsets are in place
        // units whose escapes were not staged: re-derived here (all of the
        // segment's units if more than kPackRedo)
        if (E >= 0) {
            const uint64_t lim = (uint64_t)esc_cap;
            const int nr = n_redo;
            const int64_t m = nr <= kPackRedo ? nr : s1 - s0;
            for (int64_t i = warp; i < m; i += kPackWarps) {
                const int64_t u = s0 + (nr <= kPackRedo ? redo[i] : i);
                unit_escapes(W, ldw, N, K, base, u, G, u == s0 ? E : (long long)esc_ptr[u], lim, esc, lane);
            }
        }
    }
    // 4. every offset is in place: staged escapes go out
    __syncthreads();
    if (tid == 0) {
        const bool ok = grid_barrier(esc_ptr, P - 1 + (kPackWarps + 2) * B) && sync_ok;
        sync_ok = ok;
        if (!ok) {  // reported by the caller
            st_status(esc_ptr + P, kEncTimeout);
            *reinterpret_cast<volatile int32_t *>(total) = kEncTimeout;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0) {
        esc_ptr[0] = 0;  // every block is past both barriers
        if (sync_ok) *reinterpret_cast<volatile int32_t *>(total) = __ldcg(esc_ptr + P);
    }
    if (!sync_ok) return;
    // the offsets of 32 listed units are fetched at once
    int s = 0;
    for (int i0 = 0; i0 < nl; i0 += 32) {
        int offl = -1;
        if (i0 + lane < nl) {
            const int32_t u = list_u[warp][i0 + lane];
            offl = u == 0 ? 0 : __ldcg(esc_ptr + u);
        }
        const int n = nl - i0 < 32 ? nl - i0 : 32;
        for (int j = 0; j < n; ++j) {
            const int off = __shfl_sync(kFull, offl, j);
            const int c = list_c[warp][i0 + j];
            if (off >= 0)
                for (int k = lane; k < c; k += 32)
                    if ((uint64_t)((int64_t)off + k) < (uint64_t)esc_cap) esc[(int64_t)off + k] = stage[warp][s + k];
            s += c;
        }
    }
}

// ---------------------------------------------------------------------------
// a4 / a5: decode one (stripe, group) into shared memory, apply the group's
// escapes (one thread per entry), then either store it (decode) or compare
// it with the original bits (verify).
// ---------------------------------------------------------------------------
constexpr int kStageStride = 256 + 8;  // elements; 528 bytes keeps 16-byte alignment

// Two builds: kVerify compares with W_cmp (and counts structure violations),
// else the group is stored to `out`.  The decode build fetches the group's
// escape range and each thread's first entry before decoding the planes, so
// those two dependent loads overlap the decode; it is held to 32 registers
// (eight 256-thread blocks per SM: at 35 the prefetch lost a block and was
// slower).  Verify does not prefetch (it was slower there).
template <bool kVerify>
__global__ __launch_bounds__(256, 8) void k_decode_group(TensorView t, uint16_t *__restrict__ out, int64_t ldo,
                                                      const uint16_t *__restrict__ W_cmp, int64_t ldw,
                                                      unsigned long long *__restrict__ structure_bad,
                                                      unsigned long long *__restrict__ mismatches) {
    __shared__ __align__(16) uint16_t stage[16 * kStageStride];
    const int64_t st = blockIdx.x / t.G, g = blockIdx.x % t.G, c0 = g * 4;
    const int tid = threadIdx.x;
    const int64_t u = st * t.G + g;
    int64_t p0 = 0, p1 = 0;
    uint32_t ent0 = 0u;
    if constexpr (!kVerify) {
        escape_range(t.esc_ptr, u, t.n_esc, p0, p1);
        if (p0 + tid < p1) ent0 = t.esc[p0 + tid];
    }
    {
        const int ct = tid >> 6, h = (tid >> 5) & 1, L = tid & 31;
        const int64_t c = c0 + ct;
        if (c < t.KT) {
            const uint4 hv = *reinterpret_cast<const uint4 *>(t.hi + (st * t.KT + c) * kHiTileBytes + h * 512 + L * 16);
            const uint2 lv = *reinterpret_cast<const uint2 *>(t.lo + (st * t.KT + c) * kLoTileBytes + L * 16 + h * 8);
            const int r = (L >> 2) + 8 * h;
            const int64_t n = st * 16 + r;
            const uint32_t b = (n < t.N) ? t.base[n] : 0u;
            uint32_t d[8];
            decode16(hv, lv.x, lv.y, b * 0x00800080u, d);
            uint4 *dst = reinterpret_cast<uint4 *>(stage + r * kStageStride + ct * 64 + (L & 3) * 16);
            dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
            dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
        }
    }
    __syncthreads();
    // verify also checks the escape list's structure for its group: the
    // group's offsets (and the list's first and last), each entry's key in
    // range, keys strictly increasing
    int sbad = 0;
    {
        if constexpr (kVerify) escape_range(t.esc_ptr, u, t.n_esc, p0, p1);
        for (int64_t e = p0 + tid; e < p1; e += blockDim.x) {
            const uint32_t ent = (!kVerify && e == p0 + tid) ? ent0 : t.esc[e];
            const int key = (int)(ent >> 16);
            const int r = (key >> 6) & 15, col = 64 * (key >> 10) + (key & 63);
            const bool in = key < 4096 && st * 16 + r < t.N && g * 256 + col < t.K;
            if (in) stage[r * kStageStride + col] = (uint16_t)(ent & 0xFFFFu);
            if (kVerify) sbad += (!in) + (e + 1 < p1 && (int)(t.esc[e + 1] >> 16) <= key);
        }
        if (kVerify && tid == 0) {
            const int32_t a = t.esc_ptr[u], b = t.esc_ptr[u + 1];
            sbad += (b < a) + (u == 0 && a != 0) + (u + 1 == (t.Np / 16) * t.G && (int64_t)b != t.n_esc);
        }
    }
    __syncthreads();
    const int r = tid >> 4, cc = (tid & 15) * 16;
    const int64_t n = st * 16 + r, k = c0 * 64 + cc;
    int bad = 0;
    if (n < t.N && k < t.K) {
        const uint16_t *src = stage + r * kStageStride + cc;
        const bool full = k + 16 <= t.K;
        if constexpr (!kVerify) {
            uint16_t *dst = out + n * ldo + k;
            if (full && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                reinterpret_cast<uint4 *>(dst)[0] = reinterpret_cast<const uint4 *>(src)[0];
                reinterpret_cast<uint4 *>(dst)[1] = reinterpret_cast<const uint4 *>(src)[1];
            } else {
                for (int j = 0; j < 16 && k + j < t.K; ++j) dst[j] = src[j];
            }
        } else {
            const uint16_t *w = W_cmp + n * ldw + k;
            if (full && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
                const uint4 a0 = reinterpret_cast<const uint4 *>(w)[0], a1 = reinterpret_cast<const uint4 *>(w)[1];
                const uint4 b0 = reinterpret_cast<const uint4 *>(src)[0], b1 = reinterpret_cast<const uint4 *>(src)[1];
                const uint32_t x[8] = {a0.x ^ b0.x, a0.y ^ b0.y, a0.z ^ b0.z, a0.w ^ b0.w,
                                       a1.x ^ b1.x, a1.y ^ b1.y, a1.z ^ b1.z, a1.w ^ b1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) bad += ((x[j] & 0xFFFFu) != 0) + ((x[j] >> 16) != 0);
            } else {
                for (int j = 0; j < 16 && k + j < t.K; ++j) bad += (w[j] != src[j]);
            }
        }
    }
    if constexpr (kVerify) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            bad += __shfl_xor_sync(kFull, bad, o);
            sbad += __shfl_xor_sync(kFull, sbad, o);
        }
        if ((tid & 31) == 0 && bad) atomicAdd(mismatches, (unsigned long long)bad);
        if ((tid & 31) == 0 && sbad) atomicAdd(structure_bad, (unsigned long long)sbad);
    }
}

// ---------------------------------------------------------------------------
// Escape-list structure checks.
// ---------------------------------------------------------------------------
__global__ void k_check_ptr(const int32_t *__restrict__ ptr, int64_t P, int64_t n_esc,
                            unsigned long long *__restrict__ bad) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i > P) return;
    int v = 0;
    if (i == 0 && ptr[0] != 0) ++v;
    if (i == P && (int64_t)ptr[P] != n_esc) ++v;
    if (i < P && ptr[i + 1] < ptr[i]) ++v;
    if (v) atomicAdd(bad, (unsigned long long)v);
}

}  // namespace

cudaError_t launch_encode(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, uint8_t *base, int32_t *esc_ptr,
                          uint8_t *hi, uint8_t *lo, uint32_t *esc, int64_t esc_cap, int32_t *total,
                          bool test_stall, cudaStream_t s) {
    const int64_t G = groups_of(K), P = rows_padded(N) / 16 * G;
    if (P == 0) {
        // no columns: every window holds no weight, and ties go to the
        // largest base, 239
        cudaError_t e = N > 0 ? cudaMemsetAsync(base, 239, (size_t)N, s) : cudaSuccess;
        return e != cudaSuccess ? e : cudaMemsetAsync(esc_ptr, 0, 4, s);
    }
    if (K > kLongRow)
        k_window_block<<<(unsigned)N, kRowWarps * 32, 0, s>>>(W, ldw, N, K, base, esc_ptr, P);
    else
        k_window_warp<<<(unsigned)N, 32, 0, s>>>(W, ldw, N, K, base, esc_ptr, P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the resident pack blocks, once per device (several host threads may
    // encode at once)
    static std::mutex m;
    static int slots[64] = {};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int sl = 0;
    {
        std::lock_guard<std::mutex> lock(m);
        if (dev >= 0 && dev < 64) sl = slots[dev];
        if (sl == 0) {
            int per_sm = 0, sms = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_pack, kPackWarps * 32, 0);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            sl = (per_sm > 0 ? per_sm : 1) * sms;
            if (dev >= 0 && dev < 64) slots[dev] = sl;
        }
    }
    // every block resident (the kernel has two grid barriers); the counter in
    // esc_ptr[0] must reach P - 1 + 6 B as an int32
    int64_t B = sl < P ? sl : P;
    if (P - 1 + (kPackWarps + 2) * B > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const uint8_t *cbase = base;
    int stall = test_stall ? 1 : 0;
    void *args[] = {(void *)&W, (void *)&ldw, (void *)&N, (void *)&K, (void *)&cbase, (void *)&esc_ptr,
                    (void *)&hi, (void *)&lo, (void *)&esc, (void *)&esc_cap, (void *)&P, (void *)&G,
                    (void *)&total, (void *)&stall};
    // every block must be resident at once: with fewer SMs free than the
    // occupancy query saw (another context, a partitioned device), fewer
    // blocks (longer segments) give the same result
    for (;;) {
        e = cudaLaunchCooperativeKernel((const void *)k_pack, dim3((unsigned)B), dim3(kPackWarps * 32), args, 0, s);
        if (e != cudaErrorCooperativeLaunchTooLarge || B == 1) return e;
        (void)cudaGetLastError();  // clear the launch error before the retry
        B = (B + 1) / 2;
    }
}

bool encode_timed_out(int32_t total) { return total == kEncTimeout; }

cudaError_t launch_decode(const TensorView &t, uint16_t *out, int64_t ldo, cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * t.G;
    if (blocks == 0) return cudaSuccess;
    k_decode_group<false><<<(unsigned)blocks, 256, 0, s>>>(t, out, ldo, nullptr, 0, nullptr, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_verify(const TensorView &t, const uint16_t *W, int64_t ldw, unsigned long long *structure_bad,
                          unsigned long long *count, cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * t.G;
    if (blocks == 0) return cudaSuccess;
    k_decode_group<true><<<(unsigned)blocks, 256, 0, s>>>(t, nullptr, 0, W, ldw, structure_bad, count);
    return cudaGetLastError();
}

cudaError_t launch_check_structure(const TensorView &t, int64_t esc_cap, unsigned long long *bad,
                                   cudaStream_t s) {
    (void)esc_cap;
    const int64_t P = (t.Np / 16) * t.G;
    k_check_ptr<<<(unsigned)((P + 1 + 255) / 256), 256, 0, s>>>(t.esc_ptr, P, t.n_esc, bad);
    return cudaGetLastError();
}

}  // namespace w12
