// W12 codec kernels: encode (window search, escape count, row scan, pack),
// decode, load-time verify and escape-list structure check.
//
// All of them are HBM-bound integer work (SpecPilot, arXiv 2611.02501,
// section 4.1: conversion to W12 and the bit-for-bit check of every decoded
// tensor at load time).
#include <cstdint>
#include <cstring>

#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

// ---------------------------------------------------------------------------
// a1 + a2: one warp per row.  Histogram of the exponent field over the row's
// normal finite weights, window sums over 16 consecutive exponents, argmax
// with ties to the largest base; the escape count is K minus the winning
// window's count.
// ---------------------------------------------------------------------------
constexpr int kWinWarps = 8;

__global__ __launch_bounds__(kWinWarps * 32) void k_window_count(
    const uint16_t *__restrict__ W, int64_t ldw, int64_t N, int64_t K, uint8_t *__restrict__ base,
    int32_t *__restrict__ row_ptr) {
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
        if (vec && k + 8 <= K) {
            uint4 q = *reinterpret_cast<const uint4 *>(row + k);
            memcpy(v, &q, 16);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (k + j < K) ? row[k + j] : 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = (v[j] >> 7) & 0xFF;
            const bool counted = (k + j < K) && e >= 1 && e <= 254;
            const unsigned key = counted ? (unsigned)e : 0x10000u;
            const unsigned peers = __match_any_sync(kFull, key);
            if (counted && lane == __ffs(peers) - 1) atomicAdd(&h[e], __popc(peers));
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
    if (lane == 0) {
        base[n] = (uint8_t)best_b;
        row_ptr[n + 1] = (int32_t)(K - best);
    }
}

// ---------------------------------------------------------------------------
// a2: inclusive scan of the per-row counts in row_ptr[1..N] (one block).
// row_ptr[N] = -1 flags a total that does not fit an int32 offset.
// ---------------------------------------------------------------------------
__global__ __launch_bounds__(1024) void k_row_scan(int32_t *__restrict__ row_ptr, int64_t N) {
    __shared__ long long warp_sums[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long carry = 0;
    for (int64_t c0 = 0; c0 < N; c0 += 1024) {
        const int64_t i = c0 + threadIdx.x;
        long long v = (i < N) ? (long long)row_ptr[i + 1] : 0;
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
        if (i < N) row_ptr[i + 1] = (int32_t)(incl > 0x7fffffffLL ? -1 : incl);
        carry += warp_sums[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        row_ptr[0] = 0;
        if (carry > 0x7fffffffLL) row_ptr[N] = -1;
    }
}

// ---------------------------------------------------------------------------
// a3: pack.  One block per 16-row stripe, one warp per row; each step covers
// 256 columns (4 tiles).  Records are assembled into the tile layout in
// shared memory and written out as whole tiles; escapes are written in
// column order at row_ptr[n] + rank (rank from a warp prefix sum).
// ---------------------------------------------------------------------------
__global__ __launch_bounds__(512) void k_pack(const uint16_t *__restrict__ W, int64_t ldw, int64_t N,
                                              int64_t K, const uint8_t *__restrict__ base,
                                              const int32_t *__restrict__ row_ptr,
                                              uint8_t *__restrict__ hi, uint8_t *__restrict__ lo,
                                              int32_t *__restrict__ esc_col,
                                              uint16_t *__restrict__ esc_val, int64_t esc_cap) {
    __shared__ __align__(16) uint8_t sh_hi[4 * kHiTileBytes];
    __shared__ __align__(16) uint8_t sh_lo[4 * kLoTileBytes];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x;
    const int64_t Kp = cols_padded(K), KT = Kp / 64;
    const int i = warp;  // row inside the stripe
    const int64_t n = t * 16 + i;
    const bool row_ok = n < N;
    const int b = row_ok ? base[n] : 0;
    int64_t eidx = row_ok ? row_ptr[n] : 0;
    const uint16_t *row = W + (row_ok ? n : 0) * ldw;
    const bool vec = row_ok && (reinterpret_cast<uintptr_t>(row) & 15) == 0;

    for (int64_t k0 = 0; k0 < Kp; k0 += 256) {
        const int64_t k = k0 + lane * 8;
        uint16_t v[8];
        if (vec && k + 8 <= K) {
            uint4 q = *reinterpret_cast<const uint4 *>(row + k);
            memcpy(v, &q, 16);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (row_ok && k + j < K) ? row[k + j] : 0;
        }
        uint32_t rec[8];
        unsigned emask = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = row_ok && (k + j < K);
            const int e = (v[j] >> 7) & 0xFF;
            const bool esc = in && (e == 0 || e == 255 || e < b || e > b + 15);
            if (esc) emask |= 1u << j;
            rec[j] = (in && !esc) ? (uint32_t)(((v[j] >> 15) << 11) | ((e - b) << 7) | (v[j] & 0x7F)) : 0u;
        }
        const int cnt = __popc(emask);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tmp = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += tmp;
        }
        const int total = __shfl_sync(kFull, incl, 31);
        int64_t pos = eidx + (incl - cnt);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if ((emask >> j) & 1u) {
                if (pos < esc_cap) {
                    esc_col[pos] = (int32_t)(k + j);
                    esc_val[pos] = v[j];
                }
                ++pos;
            }
        }
        eidx += total;
        if (k < Kp) {
            const int c_local = lane >> 3;
            const int jl = (lane & 7) * 8;          // column inside the tile
            const int L = (i & 7) * 4 + (jl >> 4);  // slot
            const uint32_t h0 = (rec[0] >> 4) | ((rec[1] >> 4) << 8) | ((rec[2] >> 4) << 16) | ((rec[3] >> 4) << 24);
            const uint32_t h1 = (rec[4] >> 4) | ((rec[5] >> 4) << 8) | ((rec[6] >> 4) << 16) | ((rec[7] >> 4) << 24);
            *reinterpret_cast<uint2 *>(sh_hi + c_local * kHiTileBytes + (i >> 3) * 512 + L * 16 + (jl & 15)) =
                make_uint2(h0, h1);
            uint32_t lw = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) lw |= (((rec[u] & 0xFu) << 4) | (rec[u + 4] & 0xFu)) << (8 * u);
            *reinterpret_cast<uint32_t *>(sh_lo + c_local * kLoTileBytes + L * 16 + (i >> 3) * 8 + ((jl & 15) >> 3) * 4) = lw;
        }
        __syncthreads();
        const int64_t c_first = k0 / 64;
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
    }
}

// ---------------------------------------------------------------------------
// a4 / a5: decode a (stripe, 256-column chunk) into shared memory, apply the
// escapes of the chunk, then either store it (decode) or compare it with the
// original bits (verify).
// ---------------------------------------------------------------------------
constexpr int kStageStride = 256 + 8;  // elements; 528 bytes keeps 16-byte alignment

__global__ __launch_bounds__(256) void k_decode_chunk(TensorView t, uint16_t *__restrict__ out, int64_t ldo,
                                                      const uint16_t *__restrict__ W_cmp, int64_t ldw,
                                                      unsigned long long *__restrict__ mismatches) {
    __shared__ __align__(16) uint16_t stage[16 * kStageStride];
    const int64_t nchunk = (t.KT + 3) / 4;
    const int64_t st = blockIdx.x / nchunk, c0 = (blockIdx.x % nchunk) * 4;
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
    if (tid < 16) {
        const int64_t n = st * 16 + tid;
        if (n < t.N) {
            int64_t lo, hi;
            escape_range(t.row_ptr, n, t.n_esc, lo, hi);
            const int64_t k0 = c0 * 64;
            const int64_t k1 = (k0 + 256 < t.K) ? k0 + 256 : t.K;
            for (int64_t e = lower_bound_col(t.esc_col, lo, hi, k0); e < hi; ++e) {
                const int64_t col = t.esc_col[e];
                if (col >= k1) break;
                if (col >= k0) stage[tid * kStageStride + (col - k0)] = t.esc_val[e];
            }
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
__global__ void k_check_rows(const int32_t *__restrict__ row_ptr, int64_t N, int64_t n_esc,
                             unsigned long long *__restrict__ bad) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i > N) return;
    int v = 0;
    if (i == 0 && row_ptr[0] != 0) ++v;
    if (i == N && (int64_t)row_ptr[N] != n_esc) ++v;
    if (i < N && row_ptr[i + 1] < row_ptr[i]) ++v;
    if (v) atomicAdd(bad, (unsigned long long)v);
}

__global__ void k_check_cols(TensorView t, unsigned long long *__restrict__ bad) {
    const int lane = threadIdx.x & 31;
    const int64_t n = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (n >= t.N) return;
    int64_t lo, hi;
    escape_range(t.row_ptr, n, t.n_esc, lo, hi);
    int v = 0;
    for (int64_t e = lo + lane; e < hi; e += 32) {
        const int32_t col = t.esc_col[e];
        if (col < 0 || col >= t.K) ++v;
        if (e + 1 < hi && t.esc_col[e + 1] <= col) ++v;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0 && v) atomicAdd(bad, (unsigned long long)v);
}

}  // namespace

cudaError_t launch_window_count(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, uint8_t *base,
                                int32_t *row_ptr, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int64_t blocks = (N + kWinWarps - 1) / kWinWarps;
    k_window_count<<<(unsigned)blocks, kWinWarps * 32, 0, s>>>(W, ldw, N, K, base, row_ptr);
    return cudaGetLastError();
}

cudaError_t launch_row_scan(int32_t *row_ptr, int64_t N, cudaStream_t s) {
    k_row_scan<<<1, 1024, 0, s>>>(row_ptr, N);
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, const uint8_t *base,
                        const int32_t *row_ptr, uint8_t *hi, uint8_t *lo, int32_t *esc_col,
                        uint16_t *esc_val, int64_t esc_cap, cudaStream_t s) {
    const int64_t stripes = rows_padded(N) / 16;
    if (stripes == 0 || K == 0) return cudaSuccess;
    k_pack<<<(unsigned)stripes, 512, 0, s>>>(W, ldw, N, K, base, row_ptr, hi, lo, esc_col, esc_val, esc_cap);
    return cudaGetLastError();
}

cudaError_t launch_decode(const TensorView &t, uint16_t *out, int64_t ldo, cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * ((t.KT + 3) / 4);
    if (blocks == 0) return cudaSuccess;
    k_decode_chunk<<<(unsigned)blocks, 256, 0, s>>>(t, out, ldo, nullptr, 0, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_verify(const TensorView &t, const uint16_t *W, int64_t ldw, unsigned long long *count,
                          cudaStream_t s) {
    const int64_t blocks = (t.Np / 16) * ((t.KT + 3) / 4);
    if (blocks == 0) return cudaSuccess;
    k_decode_chunk<<<(unsigned)blocks, 256, 0, s>>>(t, nullptr, 0, W, ldw, count);
    return cudaGetLastError();
}

cudaError_t launch_check_structure(const TensorView &t, int64_t esc_cap, unsigned long long *bad,
                                   cudaStream_t s) {
    (void)esc_cap;
    const int64_t b1 = (t.N + 1 + 255) / 256;
    k_check_rows<<<(unsigned)b1, 256, 0, s>>>(t.row_ptr, t.N, t.n_esc, bad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || t.N == 0) return e;
    const int64_t b2 = (t.N * 32 + 255) / 256;
    k_check_cols<<<(unsigned)b2, 256, 0, s>>>(t, bad);
    return cudaGetLastError();
}

}  // namespace w12
