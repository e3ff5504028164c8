// W12 codec kernels: encode (window search, escape count, offset scan,
// pack), decode, load-time verify and escape-list structure check.
//
// All of them are HBM-bound integer work (SpecPilot, arXiv 2611.02501,
// section 4.1: conversion to W12 and the bit-for-bit check of every decoded
// tensor at load time).  Work is organised around the 16-row x 256-column
// group, the unit the escape list is indexed by.
#include <cstdint>
#include <cstring>

#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

// Eight consecutive weights of a row, zero past K (0 is "not counted" and
// "not an escape" for the callers, which mask with k < K anyway).
__device__ __forceinline__ void load8(const uint16_t *row, bool vec, int64_t k, int64_t K, uint16_t v[8]) {
    if (vec && k + 8 <= K) {
        uint4 q = *reinterpret_cast<const uint4 *>(row + k);
        memcpy(v, &q, 16);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (k + j < K) ? row[k + j] : 0;
    }
}

// Offset-and-mantissa field of w in the window of base b: (e-b)<<7 | m, in
// [0, 0x7FF] exactly when e is in [b, b+15].  With b in [1, 239] every other
// exponent lands outside that range as an unsigned value: e = 0 and e < b
// give a negative difference, e = 255 and e > b+15 one of at least 0x800.
__device__ __forceinline__ uint32_t window_field(uint16_t w, int b) {
    return (uint32_t)((int)(w & 0x7FFF) - (b << 7));
}
__device__ __forceinline__ bool is_escape(uint16_t w, int b) { return window_field(w, b) > 0x7FFu; }

// ---------------------------------------------------------------------------
// a1 + a2: one warp per row.  Histogram of the exponent field over the row's
// normal finite weights, window sums over 16 consecutive exponents, argmax
// with ties to the largest base.  A second pass over the row counts its
// escapes per 256-column group into esc_ptr[t*G+g+1].
// ---------------------------------------------------------------------------
constexpr int kWinWarps = 8;

__global__ __launch_bounds__(kWinWarps * 32) void k_window_count(
    const uint16_t *__restrict__ W, int64_t ldw, int64_t N, int64_t K, uint8_t *__restrict__ base,
    int32_t *__restrict__ esc_ptr) {
    __shared__ int hist[kWinWarps][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kWinWarps + warp;
    if (n >= N) return;  // warp-uniform; no block-wide barrier below
    int *h = hist[warp];
    for (int i = lane; i < 256; i += 32) h[i] = 0;
    __syncwarp();
    const uint16_t *row = W + n * ldw;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    for (int64_t k0 = 0; k0 < K; k0 += 256) {
        const int64_t k = k0 + lane * 8;
        uint16_t v[8];
        load8(row, vec, k, K, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = (v[j] >> 7) & 0xFF;
            const bool counted = (k + j < K) && e >= 1 && e <= 254;
            // plain shared-memory atomics: the hardware merges lanes that hit the
            // same bin (grouping them first with __match_any_sync was 13% slower
            // over the whole encode on GB300)
            if (counted) atomicAdd(&h[e], 1);
        }
    }
    __syncwarp();
    int best = -1, best_b = 0;
    for (int b = 1 + lane; b <= 239; b += 32) {
        int c = 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) c += h[b + e];
        if (c > best || (c == best && b > best_b)) {
            best = c;
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
    if (lane == 0) base[n] = (uint8_t)best_b;
    // escapes per 256-column group (the row was just read: mostly L2 hits)
    const int64_t G = groups_of(K);
    int32_t *cnt = esc_ptr + 1 + (n / 16) * G;
    for (int64_t k0 = 0, g = 0; k0 < K; k0 += 256, ++g) {
        const int64_t k = k0 + lane * 8;
        uint16_t v[8];
        load8(row, vec, k, K, v);
        int c = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) c += (k + j < K) && is_escape(v[j], best_b);
#pragma unroll
        for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
        if (lane == 0 && c) atomicAdd(&cnt[g], c);
    }
}

// ---------------------------------------------------------------------------
// a2: inclusive scan of the per-group counts in esc_ptr[1..P] (one block).
// esc_ptr[P] = -1 flags a total that does not fit an int32 offset.
// ---------------------------------------------------------------------------
__global__ __launch_bounds__(1024) void k_ptr_scan(int32_t *__restrict__ ptr, int64_t P) {
    __shared__ long long warp_sums[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long carry = 0;
    for (int64_t c0 = 0; c0 < P; c0 += 1024) {
        const int64_t i = c0 + threadIdx.x;
        long long v = (i < P) ? (long long)ptr[i + 1] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) warp_sums[warp] = v;
        __syncthreads();
        if (warp == 0) {
            long long s = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long t = __shfl_up_sync(kFull, s, o);
                if (lane >= o) s += t;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const long long incl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + v;
        if (i < P) ptr[i + 1] = (int32_t)(incl > 0x7fffffffLL ? -1 : incl);
        carry += warp_sums[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        ptr[0] = 0;
        if (carry > 0x7fffffffLL) ptr[P] = -1;
    }
}

// ---------------------------------------------------------------------------
// a3: pack.  One block per 16-row stripe, one warp per row; each step covers
// one 256-column group (4 tiles, 8 columns per lane).  Records are assembled
// into the tile layout in shared memory and written out as whole tiles.  An
// escape at (tile c4, row i, column j) goes to
//   esc_ptr[t*G+g] + #escapes of the group before (c4,i) + rank inside (c4,i)
// with the per-(c4,i) counts exchanged through shared memory.
// ---------------------------------------------------------------------------
__global__ __launch_bounds__(512) void k_pack(const uint16_t *__restrict__ W, int64_t ldw, int64_t N,
                                              int64_t K, const uint8_t *__restrict__ base,
                                              const int32_t *__restrict__ esc_ptr,
                                              uint8_t *__restrict__ hi, uint8_t *__restrict__ lo,
                                              uint32_t *__restrict__ esc, int64_t esc_cap) {
    __shared__ __align__(16) uint8_t sh_hi[4 * kHiTileBytes];
    __shared__ __align__(16) uint8_t sh_lo[4 * kLoTileBytes];
    __shared__ int sh_cnt[2][64];  // [c4*16 + i]: counts, then exclusive prefix
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x;
    const int64_t Kp = cols_padded(K), KT = Kp / 64, G = groups_of(K);
    const int i = warp;  // row inside the stripe
    const int64_t n = t * 16 + i;
    const bool row_ok = n < N;
    const int b = row_ok ? base[n] : 0;
    const uint16_t *row = W + (row_ok ? n : 0) * ldw;
    const bool vec = row_ok && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    const int c4 = lane >> 3;         // tile inside the group
    const int jl = (lane & 7) * 8;    // first column inside the tile
    const int L = (i & 7) * 4 + (jl >> 4);  // fragment slot

    for (int64_t g = 0; g < G; ++g) {
        const int buf = (int)(g & 1);
        const int64_t k = g * 256 + lane * 8;
        uint16_t v[8];
        if (row_ok) {
            load8(row, vec, k, K, v);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0;
        }
        uint32_t rec[8];
        unsigned emask = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = row_ok && (k + j < K);
            const uint32_t f = window_field(v[j], b);
            const bool esc_ = in && f > 0x7FFu;
            if (esc_) emask |= 1u << j;
            rec[j] = (in && !esc_) ? ((uint32_t)(v[j] >> 15) << 11) | f : 0u;  // s<<11 | (e-b)<<7 | m
        }
        // per-(c4, i) count and this lane's exclusive prefix inside its 8 lanes
        const int cnt = __popc(emask);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int tmp = __shfl_up_sync(kFull, incl, o, 8);
            if ((lane & 7) >= o) incl += tmp;
        }
        if ((lane & 7) == 7) sh_cnt[buf][c4 * 16 + i] = incl;
        if (k < Kp) {
            const uint32_t h0 = (rec[0] >> 4) | ((rec[1] >> 4) << 8) | ((rec[2] >> 4) << 16) | ((rec[3] >> 4) << 24);
            const uint32_t h1 = (rec[4] >> 4) | ((rec[5] >> 4) << 8) | ((rec[6] >> 4) << 16) | ((rec[7] >> 4) << 24);
            *reinterpret_cast<uint2 *>(sh_hi + c4 * kHiTileBytes + (i >> 3) * 512 + L * 16 + (jl & 15)) =
                make_uint2(h0, h1);
            uint32_t lw = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) lw |= (((rec[u] & 0xFu) << 4) | (rec[u + 4] & 0xFu)) << (8 * u);
            *reinterpret_cast<uint32_t *>(sh_lo + c4 * kLoTileBytes + L * 16 + (i >> 3) * 8 + ((jl & 15) >> 3) * 4) = lw;
        }
        __syncthreads();
        if (warp == 0) {  // exclusive scan of the 64 counts in (c4, i) order
            const int a0 = sh_cnt[buf][2 * lane], a1 = sh_cnt[buf][2 * lane + 1];
            int s = a0 + a1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tmp = __shfl_up_sync(kFull, s, o);
                if (lane >= o) s += tmp;
            }
            const int ex = s - a0 - a1;
            sh_cnt[buf][2 * lane] = ex;
            sh_cnt[buf][2 * lane + 1] = ex + a0;
        }
        const int64_t c_first = g * 4;
        const int ntiles = (int)((KT - c_first) < 4 ? (KT - c_first) : 4);
        for (int x = threadIdx.x; x < ntiles * 96; x += blockDim.x) {
            if (x < ntiles * 64) {
                const int ct = x >> 6, o = x & 63;
                reinterpret_cast<uint4 *>(hi + (t * KT + c_first + ct) * kHiTileBytes)[o] =
                    reinterpret_cast<const uint4 *>(sh_hi + ct * kHiTileBytes)[o];
            } else {
                const int y = x - ntiles * 64;
                const int ct = y >> 5, o = y & 31;
                reinterpret_cast<uint4 *>(lo + (t * KT + c_first + ct) * kLoTileBytes)[o] =
                    reinterpret_cast<const uint4 *>(sh_lo + ct * kLoTileBytes)[o];
            }
        }
        __syncthreads();
        if (emask) {
            int64_t pos = (int64_t)esc_ptr[t * G + g] + sh_cnt[buf][c4 * 16 + i] + (incl - cnt);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if ((emask >> j) & 1u) {
                    if (pos < esc_cap)
                        esc[pos] = ((uint32_t)((c4 << 10) | (i << 6) | (jl + j)) << 16) | v[j];
                    ++pos;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// a4 / a5: decode one (stripe, group) into shared memory, apply the group's
// escapes (one thread per entry), then either store it (decode) or compare
// it with the original bits (verify).
// ---------------------------------------------------------------------------
constexpr int kStageStride = 256 + 8;  // elements; 528 bytes keeps 16-byte alignment

__global__ __launch_bounds__(256) void k_decode_group(TensorView t, uint16_t *__restrict__ out, int64_t ldo,
                                                      const uint16_t *__restrict__ W_cmp, int64_t ldw,
                                                      unsigned long long *__restrict__ mismatches) {
    __shared__ __align__(16) uint16_t stage[16 * kStageStride];
    const int64_t st = blockIdx.x / t.G, g = blockIdx.x % t.G, c0 = g * 4;
    const int tid = threadIdx.x;
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
    {
        int64_t p0, p1;
        escape_range(t.esc_ptr, st * t.G + g, t.n_esc, p0, p1);
        for (int64_t e = p0 + tid; e < p1; e += blockDim.x) {
            const uint32_t ent = t.esc[e];
            const int key = (int)(ent >> 16);
            const int r = (key >> 6) & 15, col = 64 * (key >> 10) + (key & 63);
            if (key < 4096 && st * 16 + r < t.N && g * 256 + col < t.K)
                stage[r * kStageStride + col] = (uint16_t)(ent & 0xFFFFu);
        }
    }
    __syncthreads();
    const int r = tid >> 4, cc = (tid & 15) * 16;
    const int64_t n = st * 16 + r, k = c0 * 64 + cc;
    int bad = 0;
    if (n < t.N && k < t.K) {
        const uint16_t *src = stage + r * kStageStride + cc;
        const bool full = k + 16 <= t.K;
        if (W_cmp == nullptr) {
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
    if (W_cmp != nullptr) {
#pragma unroll
        for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(kFull, bad, o);
        if ((tid & 31) == 0 && bad) atomicAdd(mismatches, (unsigned long long)bad);
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

// One warp per (stripe, group).
__global__ void k_check_entries(TensorView t, unsigned long long *__restrict__ bad) {
    const int lane = threadIdx.x & 31;
    const int64_t grp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (grp >= (t.Np / 16) * t.G) return;
    const int64_t st = grp / t.G, g = grp % t.G;
    int64_t p0, p1;
    escape_range(t.esc_ptr, grp, t.n_esc, p0, p1);
    int v = 0;
    for (int64_t e = p0 + lane; e < p1; e += 32) {
        const uint32_t key = t.esc[e] >> 16;
        const int64_t n = st * 16 + ((key >> 6) & 15), k = g * 256 + 64 * (key >> 10) + (key & 63);
        if (key >= 4096 || n >= t.N || k >= t.K) ++v;
        if (e + 1 < p1 && (t.esc[e + 1] >> 16) <= key) ++v;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0 && v) atomicAdd(bad, (unsigned long long)v);
}

}  // namespace

cudaError_t launch_window_count(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, uint8_t *base,
                                int32_t *esc_ptr, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int64_t blocks = (N + kWinWarps - 1) / kWinWarps;
    k_window_count<<<(unsigned)blocks, kWinWarps * 32, 0, s>>>(W, ldw, N, K, base, esc_ptr);
    return cudaGetLastError();
}

cudaError_t launch_ptr_scan(int32_t *esc_ptr, int64_t P, cudaStream_t s) {
    k_ptr_scan<<<1, 1024, 0, s>>>(esc_ptr, P);
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, const uint8_t *base,
                        const int32_t *esc_ptr, uint8_t *hi, uint8_t *lo, uint32_t *esc, int64_t esc_cap,
                        cudaStream_t s) {
    const int64_t stripes = rows_padded(N) / 16;
    if (stripes == 0 || K == 0) return cudaSuccess;
    k_pack<<<(unsigned)stripes, 512, 0, s>>>(W, ldw, N, K, base, esc_ptr, hi, lo, esc, esc_cap);
    return cudaGetLastError();
}

cudaError_t launch_decode(const TensorView &t, uint16_t *out, int64_t ldo, cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * t.G;
    if (blocks == 0) return cudaSuccess;
    k_decode_group<<<(unsigned)blocks, 256, 0, s>>>(t, out, ldo, nullptr, 0, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_verify(const TensorView &t, const uint16_t *W, int64_t ldw, unsigned long long *count,
                          cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * t.G;
    if (blocks == 0) return cudaSuccess;
    k_decode_group<<<(unsigned)blocks, 256, 0, s>>>(t, nullptr, 0, W, ldw, count);
    return cudaGetLastError();
}

cudaError_t launch_check_structure(const TensorView &t, int64_t esc_cap, unsigned long long *bad,
                                   cudaStream_t s) {
    (void)esc_cap;
    const int64_t P = (t.Np / 16) * t.G;
    k_check_ptr<<<(unsigned)((P + 1 + 255) / 256), 256, 0, s>>>(t.esc_ptr, P, t.n_esc, bad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || P == 0) return e;
    k_check_entries<<<(unsigned)((P * 32 + 255) / 256), 256, 0, s>>>(t, bad);
    return cudaGetLastError();
}

}  // namespace w12
