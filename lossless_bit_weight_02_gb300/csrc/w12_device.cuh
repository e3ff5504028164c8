// Device-side building blocks shared by the W12 kernels: tile geometry, the
// in-register record decoder, and small PTX wrappers.
//
// Record decode (SpecPilot, arXiv 2611.02501, section 4.1): a record
// r = s<<11 | off<<7 | m of row n becomes the BF16 bits
// s<<15 | (off+base[n])<<7 | m.  The exponent is taken modulo 256, which only
// matters for a corrupted base (a valid base is at most 239).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w12 {

constexpr int kTileRows = 16;                 // rows of one tile (one tensor-core A tile)
constexpr int kTileCols = 64;                 // columns of one tile
constexpr int kHiTileBytes = kTileRows * kTileCols;      // 1024
constexpr int kLoTileBytes = kTileRows * kTileCols / 2;  // 512
constexpr uint32_t kFull = 0xffffffffu;

__host__ __device__ inline int64_t rows_padded(int64_t N) { return (N + 15) / 16 * 16; }
__host__ __device__ inline int64_t cols_padded(int64_t K) { return (K + 255) / 256 * 256; }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Z holds, from the low byte up: a lo-plane byte whose HIGH nibble is the
// low record nibble of weight 2p, the hi byte of weight 2p, a lo-plane byte
// whose high nibble belongs to weight 2p+1, the hi byte of weight 2p+1.
// Returns the two BF16 values packed low = weight 2p, high = weight 2p+1.
//   (Z >> 4) & 0x07FF07FF  -> off<<7 | m for both halves (sign and stray
//                             nibbles dropped)
//   + base2                -> exponent off+base (no carry crosses halves:
//                             at most 270<<7|127 < 2^16)
//   select bit 15 / 31 from Z (the record signs), the rest from the sum.
__device__ __forceinline__ uint32_t decode_pair(uint32_t Z, uint32_t base2) {
    uint32_t u = ((Z >> 4) & 0x07FF07FFu) + base2;
    return (Z & 0x80008000u) | (u & 0x7FFF7FFFu);
}

// Decodes the 16 weights of one row of one tile slot: `h` is the slot's 16
// hi bytes (columns 0..15 of the slot), `l0`/`l1` its two lo words (columns
// 0..7 and 8..15).  out[p] = BF16 pair (2p, 2p+1).  base2 = base * 0x00800080.
__device__ __forceinline__ void decode16(uint4 h, uint32_t l0, uint32_t l1, uint32_t base2,
                                         uint32_t out[8]) {
    const uint32_t l0s = l0 << 4, l1s = l1 << 4;
    // columns 0..3: high nibbles of the bytes of l0; 4..7: low nibbles (l0s)
    out[0] = decode_pair(prmt(h.x, l0, 0x1504), base2);
    out[1] = decode_pair(prmt(h.x, l0, 0x3726), base2);
    out[2] = decode_pair(prmt(h.y, l0s, 0x1504), base2);
    out[3] = decode_pair(prmt(h.y, l0s, 0x3726), base2);
    out[4] = decode_pair(prmt(h.z, l1, 0x1504), base2);
    out[5] = decode_pair(prmt(h.z, l1, 0x3726), base2);
    out[6] = decode_pair(prmt(h.w, l1s, 0x1504), base2);
    out[7] = decode_pair(prmt(h.w, l1s, 0x3726), base2);
}

// Entries [lo, hi) of offset slot i (ptr[i] .. ptr[i+1]), clamped to
// [0, n_esc] so that a malformed offset can never index outside the escape
// array.
__device__ __forceinline__ void escape_range(const int32_t *__restrict__ ptr, int64_t i, int64_t n_esc,
                                             int64_t &lo, int64_t &hi) {
    int64_t a = ptr[i], b = ptr[i + 1];
    a = a < 0 ? 0 : (a > n_esc ? n_esc : a);
    b = b < a ? a : (b > n_esc ? n_esc : b);
    lo = a;
    hi = b;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

}  // namespace w12
