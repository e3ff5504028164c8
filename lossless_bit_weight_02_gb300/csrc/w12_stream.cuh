// Device helpers shared by the two W12 GEMM kernels (mma.sync and tcgen05):
// the streaming weight load, the record decoder split across the ALU and FMA
// pipes, and the per-group escape batches.
#pragma once

#include <cstdint>

#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {

// Programmatic dependent launch: a kernel may start (and prefetch its weights)
// before the previous kernel on the stream has finished; wait() returns once
// that kernel has completed and its writes are visible (a no-op when the
// launch was an ordinary one).  launch_dependents() lets the next kernel be
// scheduled.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte weight-plane load: read once, kept out of L1.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Record-pair decode (same result as decode_pair in w12_device.cuh) in four
// operations, one of them on the FMA pipe: with Z holding the two records in
// bits 4..15 and 20..31 (sign on top of each half, the neighbouring nibble
// below), clear the signs and the neighbour nibbles, then one multiply-add
// high does "shift right by 4, add base << 7" for both halves at once (no
// carry crosses a half: (base + offset) << 7 | m < 2^16 for any base byte,
// and bit 15 stays clear for the encoder's bases, which are at most 239),
// and the signs go back in.
// c28 = 2^28 arrives as a kernel argument so that it stays a multiplication.
__device__ __forceinline__ uint32_t decode_pair_fma(uint32_t Z, uint32_t base2, uint32_t c28) {
    uint32_t u;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(u) : "r"(Z & 0x7FF07FF0u), "r"(c28), "r"(base2));
    return (Z & 0x80008000u) | u;
}

__device__ __forceinline__ void decode16_fma(uint4 h, uint32_t l0, uint32_t l1, uint32_t base2, uint32_t c28,
                                             uint32_t c16, uint32_t out[8]) {
    const uint32_t l0s = l0 * c16, l1s = l1 * c16;  // << 4, on the FMA pipe
    out[0] = decode_pair_fma(prmt(h.x, l0, 0x1504), base2, c28);
    out[1] = decode_pair_fma(prmt(h.x, l0, 0x3726), base2, c28);
    out[2] = decode_pair_fma(prmt(h.y, l0s, 0x1504), base2, c28);
    out[3] = decode_pair_fma(prmt(h.y, l0s, 0x3726), base2, c28);
    out[4] = decode_pair_fma(prmt(h.z, l1, 0x1504), base2, c28);
    out[5] = decode_pair_fma(prmt(h.z, l1, 0x3726), base2, c28);
    out[6] = decode_pair_fma(prmt(h.w, l1s, 0x1504), base2, c28);
    out[7] = decode_pair_fma(prmt(h.w, l1s, 0x3726), base2, c28);
}

// silu(x) = x / (1 + e^-x) in FP32 (the fused gate/up epilogue): CUDA's
// expf and an IEEE division; -0 for very negative x, x for very large x.
__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// Fused gate/up epilogue on the tensor-core path, where lane l of a warp
// holds row 32*(warp%4) + l of a 128-row tile: the gate row 16s+i and the up
// row 16s+8+i of hidden unit 8s+i sit in lanes l and l^8.  Every lane of the
// warp must call it (a shuffle); the result is silu(gate) * up on the gate
// lanes (lane & 8 == 0), meaningless on the others.
__device__ __forceinline__ float silu_pair(float v) {
    const float up = __shfl_xor_sync(0xffffffffu, v, 8);
    return silu_f32(v) * up;
}

// Escape entries of one 256-column group, one per lane (lane < cnt).
struct EscBatch {
    uint32_t ent;  // key<<16 | BF16 bits
    int cnt;       // entries in the group (warp-uniform)
    int p0;        // index of the group's first entry (offsets are int32)
};

__device__ __forceinline__ EscBatch load_group_escapes(const TensorView &t, int p0, int p1, int lane) {
    EscBatch b;
    b.p0 = p0;
    b.cnt = (int)(p1 - p0);
    b.ent = (lane < b.cnt) ? __ldg(t.esc + p0 + lane) : 0u;
    return b;
}

// Bit p set when tile p of the group holds an escape (all bits when the group
// holds more than 32, which are then walked from memory).
__device__ __forceinline__ uint32_t escape_tiles(const EscBatch &b, int lane) {
    if (b.cnt > 32) return 0xFu;
    const uint32_t c4 = b.ent >> 26;
    const uint32_t bit = (lane < b.cnt && c4 < 4) ? (1u << c4) : 0u;
    return __reduce_or_sync(kFull, bit);
}

// Ranges: work units are cut into segments of g.seglen units (the whole
// tensor, or one stripe / row tile), and each segment into g.per contiguous
// ranges: the first g.rem ranges of a segment hold g.q + 1 units, the others
// g.q.  The small-M kernel numbers its units u = stripe*G + group, the
// tensor-core kernel u = row_tile*G + group; both planes and the escape
// offsets are stored stripe-major with whole groups, so a range is one
// contiguous stream however many stripe boundaries it crosses.  All of it
// is 32-bit integer arithmetic (unit and range counts are below 2^31).
__device__ __forceinline__ int range_begin(int v, const GemmArgs &g) {
    const int seg = v / g.per, j = v - seg * g.per;
    return seg * g.seglen + j * g.q + (j < g.rem ? j : g.rem);
}
// the range holding unit u
__device__ __forceinline__ int range_of(int u, const GemmArgs &g) {
    const int seg = u / g.seglen, x = u - seg * g.seglen;
    const int big = g.rem * (g.q + 1);  // units in the segment's longer ranges
    const int j = x < big ? x / (g.q + 1) : g.rem + (x - big) / g.q;
    return seg * g.per + j;
}

}  // namespace w12
