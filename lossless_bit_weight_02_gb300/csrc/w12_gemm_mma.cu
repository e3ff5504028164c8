// Small-M W12 GEMM (1 <= M <= 16): Y = A * W^T with the weights decoded in
// registers (SpecPilot, arXiv 2611.02501, section 4.1: "decodes records in
// registers", "splits the reduction in a fixed order so the GEMM is
// deterministic").
//
// Design (HBM-bound: ~1.33*M flop per weight byte):
//   * Work: the (16-row stripe, 256-column group) units, in stripe-major
//     order, are cut into one contiguous range per resident warp, so every
//     warp streams the same number of groups whatever the stripe count; a
//     range may start and end inside stripes.  Each warp streams its range's
//     tiles: per 16x64 tile every lane issues two 128-bit
//     loads of the hi plane and one of the lo plane - the tile layout puts
//     exactly the lane's tensor-core A fragment (rows g and g+8, 16 columns
//     each) behind those loads, so a warp reads 1.5 KB contiguous per tile.
//   * Records are decoded to BF16 pairs with two integer ops per weight
//     (prmt / and / multiply-add-high / select per pair), escapes of the
//     tile are patched in (through a 2 KB per-warp shared-memory copy of the
//     fragment, only for tiles that hold an escape), then four
//     mma.sync.m16n8k16 per 8 tokens accumulate in FP32.  The 64 columns of
//     a tile are fed to the four MMAs in a fixed permuted order; activations
//     use the same permutation.
//   * Activations: every warp copies the next group's 256 columns of the
//     token rows into its own shared-memory buffer with cp.async while it
//     works on the current group, so the B fragments come from shared memory
//     (the warps of an SM would otherwise all wait on the same L2 lines).
//   * Fixed-order reduction: a stripe that lies inside one range is rounded
//     and stored directly; the pieces of a stripe cut by range boundaries go
//     to an FP32 workspace, and the warp delivering the last piece sums them
//     in range order and writes BF16.  The cut depends on (M, N, K) only, so
//     the result is identical for any grid.
#include <cstdint>
#include <mutex>

#include "w12_device.cuh"
#include "w12_internal.h"
#include "w12_stream.cuh"

namespace w12 {
namespace {

// Warps per block, each keeping one 4-tile group in flight: a whole SM's
// worth (16 for M <= 8, 12 for M <= 16, which is what the registers and the
// shared memory allow) in one block.  The warp scheduler favours older
// blocks: with four 4-warp blocks per SM, the youngest block's warps streamed
// their ranges ~20% slower than the oldest's, and each SM ended its launch
// with few warps left.  The warps of one block run at the same pace.
template <int NB>
__host__ __device__ constexpr int warps_of() {
    return NB == 1 ? 16 : 12;
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Activations are staged in shared memory a whole 256-column group ahead:
// each warp owns two buffers of 8*NB token rows x kActPitch BF16 (the 8
// padding columns put the rows of one 8-lane phase on different banks, so
// the fragment reads below are conflict-free).
constexpr int kActPitch = 264;

template <int NB>
__host__ __device__ constexpr uint32_t act_buf_bytes() {
    return 8 * NB * kActPitch * 2;
}
template <int NB>
__host__ __device__ constexpr int smem_bytes() {
    return warps_of<NB>() * (4 * 32 * 16 + 2 * act_buf_bytes<NB>());
}

// CG: cache the copy in L2 only (activations another SM has just written,
// in a list of dependent GEMMs); otherwise in L1 too.
template <bool CG>
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    if (CG)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Copies columns 256*gg .. 256*gg+255 of the first `rows` token rows of A into
// the buffer at shared address `dst`: lane l takes columns 8l .. 8l+7 of each
// row (16 bytes; A rows are 16-byte aligned).  Columns at or beyond K read as
// zero.
template <int NB, bool CG>
__device__ __forceinline__ void stage_group(uint32_t dst, const uint16_t *__restrict__ A, int64_t lda, int rows,
                                            int64_t gg, int64_t K, int lane) {
    const int64_t col = gg * 256 + 8 * lane;
    const int64_t rem = K - col;
    const uint32_t bytes = rem >= 8 ? 16u : (rem > 0 ? (uint32_t)rem * 2u : 0u);
    const uint16_t *src = bytes ? A + col : A;
    const int64_t step = bytes ? lda : 0;
#pragma unroll
    for (int i = 0; i < 8 * NB; ++i)
        if (i < rows) cp_async16<CG>(dst + (uint32_t)(i * kActPitch + 8 * lane) * 2u, src + i * step, bytes);
    cp_async_commit();
}


__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds128s(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// Byte of weight (row r, column j) of a 16x64 tile in the per-warp copy of
// the A fragments ([4][32] uint4: pair group (j%16)/4, slot 4*(r%8) + j/16,
// component ((j%16)/2 & 1)*2 + r/8, half j&1).
__device__ __forceinline__ uint32_t patch_byte(uint32_t r, uint32_t j) {
    const uint32_t slot = (r & 7) * 4 + (j >> 4), j16 = j & 15, pr = j16 >> 1;
    const uint32_t comp = (pr & 1) * 2 + (r >> 3);
    return ((pr >> 1) * 32 + slot) * 16 + comp * 4 + (j16 & 1) * 2;
}

// Writes escape `ent` (key<<16 | bits) into the per-warp fragment copy at
// shared address `patch`.
__device__ __forceinline__ void patch_one(uint32_t patch, uint32_t ent, uint32_t vmask) {
    const uint32_t key = ent >> 16;
    const uint16_t val = (uint16_t)(ent & vmask);
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(patch + patch_byte((key >> 6) & 15, key & 63)), "h"(val)
                 : "memory");
}

// Per-warp streaming state of one work item.  (Kept small: the 16-warp
// build runs at its 128-register limit.)
template <int NB>
struct Stream {
    uint4 bh0[4], bh1[4], bl[4];  // the 4 tiles of the current group (prefetched)
    uint32_t hidx;                // uint4 index of this lane's hi-plane bytes of the current group:
                                  // 256 * unit + lane (its lo-plane index is (hidx + lane) / 2)
    uint32_t base2A, base2B;      // row bases * 0x00800080 (rows g, g+8)
    float acc[NB][4];
    EscBatch cur;                 // escapes of the current group
    uint32_t emask;               // tiles of the group holding an escape
    uint32_t esc1;                // this lane's escape: bits | byte in the fragment copy << 16 | tile << 27
};

// One unit u (a 256-column group of one stripe): stage the next unit's
// activations (column group gnext), then for each of the 4 tiles read the B
// fragments from shared memory, decode the two rows, prefetch the same tile
// of the next unit (or, on the last unit, the same tile again: an L2 hit),
// patch the tile's escapes and run the MMAs.  Q: the nested 8-bit view (the
// lo plane is neither loaded nor used; escape values lose their 4 low
// mantissa bits).
template <int NB, bool Q, bool CG>
__device__ __forceinline__ void group_step(Stream<NB> &w, const TensorView &t, const GemmArgs &g, int u,
                                           int gnext, bool more, uint32_t patch, int lane,
                                           int rows, uint32_t act, uint32_t frag,
                                           uint32_t c28, uint32_t c16) {
    // This lane's copies for unit u have landed; after the warp barrier so
    // have every lane's, and every lane is done reading the other buffer.
    cp_async_wait_all();
    __syncwarp();
    if (more) stage_group<NB, CG>(act + (uint32_t)((u + 1) & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, gnext, t.K, lane);
    const uint32_t ab = act + (uint32_t)(u & 1) * act_buf_bytes<NB>() + frag;
    // the next group's tiles (on the last unit, the same tiles again: L2 hits)
    const uint4 *hp = reinterpret_cast<const uint4 *>(t.hi) + w.hidx + (more ? 256 : 0);
    const uint4 *lp = reinterpret_cast<const uint4 *>(t.lo) + ((w.hidx + lane) >> 1) + (more ? 128 : 0);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t bw[NB][8];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t a = ab + (uint32_t)(8 * b * kActPitch + 64 * p) * 2u;
            const uint4 v0 = lds128s(a), v1 = lds128s(a + 16);
            bw[b][0] = v0.x; bw[b][1] = v0.y; bw[b][2] = v0.z; bw[b][3] = v0.w;
            bw[b][4] = v1.x; bw[b][5] = v1.y; bw[b][6] = v1.z; bw[b][7] = v1.w;
        }
        uint32_t dA[8], dB[8];
        if (Q) {
            decode16_fma(w.bh0[p], 0u, 0u, w.base2A, c28, c16, dA);
            decode16_fma(w.bh1[p], 0u, 0u, w.base2B, c28, c16, dB);
        } else {
            decode16_fma(w.bh0[p], w.bl[p].x, w.bl[p].y, w.base2A, c28, c16, dA);
            decode16_fma(w.bh1[p], w.bl[p].z, w.bl[p].w, w.base2B, c28, c16, dB);
        }
        w.bh0[p] = ld_stream(hp + p * 64);
        w.bh1[p] = ld_stream(hp + p * 64 + 32);
        if (!Q) w.bl[p] = ld_stream(lp + p * 32);

        // Escapes of this tile replace the decoded placeholders.
        if ((w.emask >> p) & 1u) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sts128(patch + (uint32_t)(i * 32 + lane) * 16u, make_uint4(dA[2 * i], dB[2 * i], dA[2 * i + 1], dB[2 * i + 1]));
            __syncwarp();
            if (w.cur.cnt <= 32) {
                asm volatile("{\n.reg .pred pp;\nsetp.eq.u32 pp, %0, %1;\n@pp st.shared.u16 [%2], %3;\n}" ::"r"(w.esc1 >> 27),
                             "r"((uint32_t)p), "r"(patch + ((w.esc1 >> 16) & 0x7FFu)), "h"((uint16_t)w.esc1)
                             : "memory");
            } else {  // more than 32 escapes in the group: walk it in batches
                for (int b0 = 0; b0 < w.cur.cnt; b0 += 32) {
                    const uint32_t e = (b0 + lane < w.cur.cnt) ? __ldg(t.esc + w.cur.p0 + b0 + lane) : 0u;
                    if (b0 + lane < w.cur.cnt && (int)(e >> 26) == p) patch_one(patch, e, Q ? 0xFFF0u : 0xFFFFu);
                }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = lds128s(patch + (uint32_t)(i * 32 + lane) * 16u);
                dA[2 * i] = v.x;
                dB[2 * i] = v.y;
                dA[2 * i + 1] = v.z;
                dB[2 * i + 1] = v.w;
            }
            __syncwarp();
        }

#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
                mma16816(w.acc[b], dA[2 * i], dB[2 * i], dA[2 * i + 1], dB[2 * i + 1], bw[b][2 * i],
                         bw[b][2 * i + 1]);
        }
    }
}

// This lane's escape of the current group (at most one while the group holds
// <= 32): its tile, its byte in the per-warp fragment copy (slot
// 4*(row%8)+col/16, component (pair&1)*2+row/8, half col&1), its bits.
template <int NB, bool Q>
__device__ __forceinline__ void own_escape(Stream<NB> &w, int lane) {
    w.emask = escape_tiles(w.cur, lane);
    w.esc1 = 4u << 27;  // tile 4: no escape for this lane
    if (lane < w.cur.cnt && w.cur.cnt <= 32) {
        const uint32_t key = w.cur.ent >> 16;
        w.esc1 = (w.cur.ent & (Q ? 0xFFF0u : 0xFFFFu)) | patch_byte((key >> 6) & 15, key & 63) << 16 | (key >> 10) << 27;
    }
}

// What one warp of a small-M kernel keeps for every range it streams: its
// shared-memory areas and lane geometry.
template <int NB>
struct WarpCtx {
    uint32_t patch;               // shared address of the warp's 2 KB escape-patch copy
    uint32_t act;                 // shared address of the warp's two activation buffers
    uint32_t frag;                // this lane's fragment offset inside a buffer
    int lane, gid, q;
    uint32_t c28, c16;
};

// Range v of the GEMM (t, g): units [range_begin(v), range_begin(v+1)) in
// stripe-major order.  Streams the range's tiles, stores every stripe that
// lies inside the range, hands the pieces of stripes cut by range boundaries
// to the FP32 slots and, if this warp delivers a stripe's last piece, sums
// them in range order and stores the stripe.  before_reads() runs once,
// after the range's first weights and escapes are in flight and before the
// first read of A, Y or the workspace.  With g.silu the stored value of
// hidden unit 8*stripe + i is silu(row 16*stripe + i) * (row 16*stripe + 8 + i).
template <int NB, bool Q, bool CG, class BeforeReads>
__device__ __forceinline__ void mma_range(const TensorView &t, const GemmArgs &g, int v, const WarpCtx<NB> &c,
                                          BeforeReads &&before_reads) {
    constexpr int MP = 8 * NB;
    constexpr int kSlot = 16 * MP;  // floats in one partial (16 rows x MP tokens)
    const int lane = c.lane, gid = c.gid, q = c.q;
    const int G = (int)t.G;  // unit indices fit an int32 (checked on the host)
    const int rows = g.M < MP ? (int)g.M : MP;  // staged token rows
    const uint4 *hi4 = reinterpret_cast<const uint4 *>(t.hi);
    const uint4 *lo4 = reinterpret_cast<const uint4 *>(t.lo);
    const int n_esc = (int)t.n_esc;  // offsets are int32
    const int ranges = (int)g.ranges;

    const int u0 = range_begin(v, g), u1 = range_begin(v + 1, g);
    if (u0 >= u1) {  // (the automatic and forced cuts make none; before_reads still runs once)
        before_reads();
        return;
    }
    const int nu = (int)(u1 - u0);  // units in the range
    Stream<NB> w;

    // 1. weight stream first, so that its latency covers the set-up below
    w.hidx = (uint32_t)u0 * 256u + (uint32_t)lane;  // fits: the host limits a tensor to 2^24 units
    {
        const uint4 *hp = hi4 + w.hidx, *lp = lo4 + (uint32_t)u0 * 128u + (uint32_t)lane;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            w.bh0[p] = ld_stream(hp + p * 64);
            w.bh1[p] = ld_stream(hp + p * 64 + 32);
            if (!Q) w.bl[p] = ld_stream(lp + p * 32);
        }
    }
    // 2. the first stripe's bases, escape offsets (lane l holds the
    //    offset of unit u0 + iw0 + l), escapes of the first two units
    int st = u0 / G;
    int gi = u0 - st * G;  // group of unit u in its stripe
    auto bases = [&](int stripe, uint32_t &bA, uint32_t &bB) {
        const int rA = stripe * 16 + gid, rB = rA + 8;
        bA = (rA < t.N ? (uint32_t)__ldg(t.base + rA) : 0u) * 0x00800080u;
        bB = (rB < t.N ? (uint32_t)__ldg(t.base + rB) : 0u) * 0x00800080u;
    };
    bases(st, w.base2A, w.base2B);
    const int32_t *gptr = t.esc_ptr + u0;
    int iw0 = 0;
    auto load_window = [&](int first) -> int {
        const int i = first + lane;
        int x = 0;
        if (i <= nu) {
            x = __ldg(gptr + i);
            x = x < 0 ? 0 : (x > n_esc ? n_esc : x);
        }
        return x;
    };
    int ptrw = load_window(0);
    auto unit_bounds = [&](int i, int &p0, int &p1) {
        if (i + 1 - iw0 >= 32) {  // slide the window (more than 30 units per range)
            iw0 = i;
            ptrw = load_window(iw0);
        }
        p0 = __shfl_sync(kFull, ptrw, i - iw0);
        p1 = __shfl_sync(kFull, ptrw, i + 1 - iw0);
        if (p1 < p0) p1 = p0;
    };
    int p0 = 0, p1 = 0;
    EscBatch nxt;
    nxt.cnt = 0;
    nxt.ent = 0;
    nxt.p0 = 0;
    unit_bounds(0, p0, p1);
    w.cur = load_group_escapes(t, p0, p1, lane);
    if (nu > 1) {
        unit_bounds(1, p0, p1);
        nxt = load_group_escapes(t, p0, p1, lane);
    }

    // Everything above reads only the W12 tensor; activations, Y and the
    // workspace may belong to earlier work.
    before_reads();

    // every lane is done with the buffers of this warp's previous range
    __syncwarp();
    stage_group<NB, CG>(c.act + (uint32_t)(u0 & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, gi, t.K, lane);
    own_escape<NB, Q>(w, lane);

    // Arrival counts still to be read: lane 0's count for the range's
    // first piece when later units follow (-1: none; its stripe is the
    // one holding u0), and for the range's last piece.
    int pend_old = -1, last_old = 0;
    int last_st = -1;
    int i = 0;  // units of the range done
    // One stripe piece per pass: units [u0 + i, u0 + pe) of stripe st.
    while (i < nu) {
        const int piece0 = u0 + i;
        const int pe = (st + 1) * G - u0 < nu ? (st + 1) * G - u0 : nu;
        // Token rows beyond M are never staged: whatever their buffer rows
        // hold only reaches accumulator columns that are never stored.
#pragma unroll
        for (int b = 0; b < NB; ++b) w.acc[b][0] = w.acc[b][1] = w.acc[b][2] = w.acc[b][3] = 0.f;
        for (; i < pe; ++i) {
            const bool more = i + 1 < nu;
            group_step<NB, Q, CG>(w, t, g, u0 + i, gi + 1 == G ? 0 : gi + 1, more, c.patch, lane, rows, c.act,
                                  c.frag, c.c28, c.c16);
            w.hidx += 256;
            ++gi;
            // the next unit's escapes are already in flight; fetch the one after
            w.cur = nxt;
            if (more) own_escape<NB, Q>(w, lane);
            if (i + 2 < nu) {
                unit_bounds(i + 2, p0, p1);
                nxt = load_group_escapes(t, p0, p1, lane);
            }
        }

        // The piece [piece0, u0 + pe) of stripe st ends here.
        // acc[b] = {(rowA, m0), (rowA, m0+1), (rowB, m0), (rowB, m0+1)}, m0 = 8b + 2q.
        const int n0 = st * 16, sbeg = st * G;
        const int rowA = n0 + gid, rowB = n0 + gid + 8;
        const bool more = i < nu;
        if (piece0 == sbeg && gi == G) {  // the whole stripe: round and store
#pragma unroll
            for (int b = 0; b < NB; ++b) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 8 * b + 2 * q + h;
                    if (m < g.M) {
                        if (g.silu) {
                            g.Y[(int64_t)m * g.ldy + st * 8 + gid] =
                                f32_to_bf16_rn(silu_f32(w.acc[b][h]) * w.acc[b][2 + h]);
                        } else {
                            if (rowA < t.N) g.Y[(int64_t)m * g.ldy + rowA] = f32_to_bf16_rn(w.acc[b][h]);
                            if (rowB < t.N) g.Y[(int64_t)m * g.ldy + rowB] = f32_to_bf16_rn(w.acc[b][2 + h]);
                        }
                    }
                }
            }
        } else {
            // Partial: slot v for the range's first piece, v + ranges for
            // a later one.  The arrival count is read only at the end of
            // the range, so the atomic's round trip never stalls the
            // stream; the last of the stripe's pieces to arrive then sums
            // them in range order and stores.
            float *slot = g.partials + ((int64_t)v + (piece0 == u0 ? 0 : ranges)) * kSlot;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                *reinterpret_cast<float2 *>(slot + gid * MP + 8 * b + 2 * q) = make_float2(w.acc[b][0], w.acc[b][1]);
                *reinterpret_cast<float2 *>(slot + (gid + 8) * MP + 8 * b + 2 * q) =
                    make_float2(w.acc[b][2], w.acc[b][3]);
            }
            __threadfence();
            __syncwarp();
            int old = 0;
            if (lane == 0) old = atomicAdd(&g.counters[st], 1);
            if (piece0 == u0 && more) {
                pend_old = old;
            } else {
                last_st = st;
                last_old = old;
            }
        }
        if (more) {  // on to the next stripe (its first unit's weights are in flight already)
            ++st;
            gi = 0;
            bases(st, w.base2A, w.base2B);
        }
    }

    // Stripes whose last piece this warp delivered: sum their partials.
    pend_old = __shfl_sync(kFull, pend_old, 0);
    for (int k = 0; k < 2; ++k) {
        const int rs = k == 0 ? (pend_old >= 0 ? u0 / G : -1) : last_st;
        if (rs < 0) continue;
        const int sbeg = rs * G;
        const int va = range_of(sbeg, g), vb = range_of(sbeg + G - 1, g);
        const int fin = __shfl_sync(kFull, (k == 0 ? pend_old : last_old) == (int)(vb - va), 0);
        if (!fin) continue;
        __threadfence();
        // only range va can start before the stripe (its piece is then a later one)
        const float *first = g.partials + ((int64_t)va + (range_begin(va, g) < sbeg ? ranges : 0)) * kSlot;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float2 sum[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int lr = gid + 8 * rr;
                const int off = lr * MP + 8 * b + 2 * q;
                sum[rr] = __ldcg(reinterpret_cast<const float2 *>(first + off));
                for (int x = va + 1; x <= vb; x += 4) {  // four independent loads at a time
                    float2 y[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (x + j <= vb)
                            y[j] = __ldcg(reinterpret_cast<const float2 *>(g.partials + (int64_t)(x + j) * kSlot + off));
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (x + j <= vb) {
                            sum[rr].x += y[j].x;
                            sum[rr].y += y[j].y;
                        }
                }
            }
            const int m = 8 * b + 2 * q;
            if (g.silu) {
                const int col = rs * 8 + gid;
                if (m < g.M) g.Y[(int64_t)m * g.ldy + col] = f32_to_bf16_rn(silu_f32(sum[0].x) * sum[1].x);
                if (m + 1 < g.M) g.Y[(int64_t)(m + 1) * g.ldy + col] = f32_to_bf16_rn(silu_f32(sum[0].y) * sum[1].y);
            } else {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = rs * 16 + gid + 8 * rr;
                    if (row < t.N) {
                        if (m < g.M) g.Y[(int64_t)m * g.ldy + row] = f32_to_bf16_rn(sum[rr].x);
                        if (m + 1 < g.M) g.Y[(int64_t)(m + 1) * g.ldy + row] = f32_to_bf16_rn(sum[rr].y);
                    }
                }
            }
        }
        if (lane == 0) g.counters[rs] = 0;
    }
}

template <int NB>
__device__ __forceinline__ WarpCtx<NB> warp_ctx(unsigned char *smem, int warp, int lane, uint32_t c28, uint32_t c16) {
    constexpr int kWarps = warps_of<NB>();
    WarpCtx<NB> c;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem);
    c.patch = base + (uint32_t)warp * 2048u;
    c.act = base + kWarps * 2048u + (uint32_t)warp * 2u * act_buf_bytes<NB>();
    c.lane = lane;
    c.gid = lane >> 2;
    c.q = lane & 3;
    c.frag = (uint32_t)(c.gid * kActPitch + 16 * c.q) * 2u;
    c.c28 = c28;
    c.c16 = c16;
    return c;
}

template <int NB, bool Q>  // NB = number of 8-token column blocks (1: M <= 8, 2: M <= 16); Q: nested 8-bit view
__global__ __launch_bounds__(warps_of<NB>() * 32, 1) void k_gemm_mma(TensorView t, GemmArgs g) {
    constexpr int kWarps = warps_of<NB>();
    // [kWarps][4][32] uint4 escape-patch copies, then [kWarps][2][8*NB][kActPitch] activations
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WarpCtx<NB> c = warp_ctx<NB>(smem, warp, lane, g.c28, g.c16);
    grid_dep_launch();
    bool dep_done = false;
    const int ranges = (int)g.ranges;
    for (int v = blockIdx.x * kWarps + warp; v < ranges; v += gridDim.x * kWarps)
        mma_range<NB, Q, false>(t, g, v, c, [&] {
            if (!dep_done) {
                grid_dep_wait();
                dep_done = true;
            }
        });
}

// ---- a list of GEMMs in one persistent launch ----

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t x;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(x));
    return x;
}

// Waits (every lane) until *count reaches `target`.  Bounded: after about a
// second (or 2^22 polls) it records W12_ERR_TIMEOUT in the error word and
// returns, so a broken dependency can never hang the GPU.
__device__ __forceinline__ void wait_count(const int32_t *count, int target, int32_t *err) {
    if (ld_acquire(count) >= target) return;
    const uint64_t t0 = global_timer_ns();
    for (int i = 1; i < (1 << 22); ++i) {
        __nanosleep(64);
        if (ld_acquire(count) >= target) return;
        if ((i & 15) == 0 && global_timer_ns() - t0 > 1000000000ull) break;
    }
    atomicExch(err, 1);
}

// Whether phase 0 of the shared-memory mbarrier at `bar` has completed
// (try_wait may suspend the thread for a short, hardware-chosen time).
__device__ __forceinline__ bool mbar_test(uint32_t bar) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\nselp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(bar)
                 : "memory");
    return ok != 0;
}

// Waits until phase 0 of the mbarrier at `bar` completes (another warp of the
// block arrives on it); bounded like wait_count.
__device__ __forceinline__ void mbar_wait_bounded(uint32_t bar, int32_t *err) {
    if (mbar_test(bar)) return;
    const uint64_t t0 = global_timer_ns();
    for (int i = 1; i < (1 << 22); ++i) {
        if (mbar_test(bar)) return;
        if ((i & 15) == 0 && global_timer_ns() - t0 > 1000000000ull) break;
    }
    atomicExch(err, 1);
}

// The GEMMs of the list one after another on one grid of resident warps:
// warp W takes ranges W, W + total warps, ... of every GEMM in list order,
// with each GEMM's own cut (the one w12_gemm uses), so every result is
// bitwise the one w12_gemm gives.  A warp reads a GEMM's activations only
// after the GEMM it names in `after` has completed (all its ranges counted
// in done[]), and uses a slice of FP32 slots and arrival counters only after
// the GEMM kListSlices earlier, which used the same slice, has completed.  No
// warp waits for a later GEMM, so with every warp resident (a cooperative
// launch) the waits always end.  One warp per block polls a count in global
// memory; the block's other warps wait on a shared-memory mbarrier it
// arrives on (with every warp of the grid polling one address, the polls
// slowed the very increments they waited for: 7.7 us per dependent GEMM on
// GB300).  The last warp to finish clears done[].
template <int NB, bool Q>
__global__ __launch_bounds__(warps_of<NB>() * 32, 1) void k_gemm_mma_list(const __grid_constant__ ListParams lp) {
    constexpr int kWarps = warps_of<NB>();
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WarpCtx<NB> c = warp_ctx<NB>(smem, warp, lane, lp.c28, lp.c16);
    // Per count waited for (slot kListMax: the stall test's): an mbarrier
    // whose phase 0 completes when the block's polling warp has seen the
    // count reached, and whether a warp of the block is polling it.
    __shared__ __align__(8) uint64_t sh_seen[kListMax + 1];
    __shared__ int sh_poll[kListMax + 1];
    for (int i = threadIdx.x; i <= kListMax; i += blockDim.x) {
        sh_poll[i] = 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(sh_seen + i))
                     : "memory");
    }
    __syncthreads();
    grid_dep_launch();
    bool dep_done = false;
    const int W = blockIdx.x * kWarps + warp, TW = gridDim.x * kWarps;
    auto block_wait = [&](int slot, const int32_t *count, int target) {
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(sh_seen + slot);
        if (!mbar_test(bar)) {
            int poller = 0;
            if (lane == 0) poller = atomicCAS(sh_poll + slot, 0, 1) == 0;
            if (__shfl_sync(kFull, poller, 0)) {
                wait_count(count, target, lp.error);  // acquire at GPU scope
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
            } else {
                mbar_wait_bounded(bar, lp.error);  // suspended in hardware between polls
            }
        }
        // a GPU-scope fence in every warp before it reads what the count
        // covered (the activations are staged through L1, cp.async.ca: at
        // M = 16 that was 9% faster than L2-only copies)
        __threadfence();
        __syncwarp();
    };
    for (int i = 0; i < lp.n; ++i) {
        // references into the parameter space, not copies: the compiler then
        // reloads a field where it needs it instead of spilling a copy (the
        // 12-warp build went from 80 bytes of spills to none)
        const TensorView &t = lp.item[i].t;
        const GemmArgs &g = lp.item[i].g;
        bool waited = false;
        for (int v = W; v < (int)g.ranges; v += TW) {
            mma_range<NB, Q, false>(t, g, v, c, [&] {
                if (waited) return;
                waited = true;
                if (!dep_done) {
                    grid_dep_wait();
                    dep_done = true;
                }
                const int a = lp.item[i].after;
                if (a >= 0) block_wait(a, lp.done + a, (int)lp.item[a].g.ranges);
                // tests of the bounded wait: a count no warp can complete
                // while this one waits (it has not exited)
                if (a == -2) block_wait(kListMax, lp.exit_count, TW + 1);
                const int r = i - kListSlices;
                if (r >= 0) block_wait(r, lp.done + r, (int)lp.item[r].g.ranges);
            });
            // the range's stores (and any stripe sums it made) come first
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(lp.done + i, 1);
        }
    }
    __syncwarp();
    if (lane == 0 && atomicAdd(lp.exit_count, 1) == TW - 1) {
        // every warp has finished all its waits: clear the counts for the next launch
        for (int i = 0; i < lp.n; ++i) lp.done[i] = 0;
        *lp.exit_count = 0;
        __threadfence();
    }
}

// Per device: SM count and, per kernel build, its occupancy (set up once,
// under a lock: several host threads may launch at once).
struct LaunchCache {
    int sms = 0;
    int occ[2][3][2] = {};  // [list kernel][NB][Q]
};
std::mutex g_launch_mutex;

template <class Kern>
cudaError_t launch_setup(Kern kern, int list, int nb, bool q, int threads, int smem, int &sms, int &occ) {
    static LaunchCache caches[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_launch_mutex);
    LaunchCache &lc = caches[dev & 63];
    if (lc.sms == 0) {
        e = cudaDeviceGetAttribute(&lc.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    int &slot = lc.occ[list][nb][q ? 1 : 0];
    if (slot == 0) {
        int o = 0;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem);
        if (e != cudaSuccess) return e;
        slot = o > 0 ? o : 1;
    }
    sms = lc.sms;
    occ = slot;
    return cudaSuccess;
}

template <int NB, bool Q>
cudaError_t launch_nb(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    constexpr int kWarps = warps_of<NB>();
    int sms = 0, occ = 0;
    cudaError_t e = launch_setup(k_gemm_mma<NB, Q>, 0, NB, Q, kWarps * 32, smem_bytes<NB>(), sms, occ);
    if (e != cudaSuccess) return e;
    int64_t blocks = (g.ranges + kWarps - 1) / kWarps;
    const int64_t resident = (int64_t)sms * occ;
    if (blocks > resident) blocks = resident;
    if (g.max_ctas > 0 && blocks > g.max_ctas) blocks = g.max_ctas;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem_bytes<NB>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemm_mma<NB, Q>, t, g);
}

// One persistent, cooperative launch (every block resident, which the
// dependency waits rely on) over the list's GEMMs.
template <int NB, bool Q>
cudaError_t launch_list_nb(const ListParams &lp, int max_ctas, bool overlap, cudaStream_t s) {
    constexpr int kWarps = warps_of<NB>();
    int sms = 0, occ = 0;
    cudaError_t e = launch_setup(k_gemm_mma_list<NB, Q>, 1, NB, Q, kWarps * 32, smem_bytes<NB>(), sms, occ);
    if (e != cudaSuccess) return e;
    int64_t blocks = (int64_t)sms * occ;
    if (max_ctas > 0 && blocks > max_ctas) blocks = max_ctas;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem_bytes<NB>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k_gemm_mma_list<NB, Q>, lp);
}

}  // namespace

int64_t gemm_mma_partial_cols(int64_t M) { return M <= 8 ? 8 : 16; }

// The range cut depends on (M, N, K, split_k) only, never on the grid, so
// the summation order (and the result) is the same for any launch.
//  * automatic: one range per resident warp of a 152-SM GPU (16 warps per
//    SM for M <= 8, 12 for M <= 16) over the whole tensor, so that every
//    warp streams the same number of groups whatever the stripe count; at
//    most one range per unit.
//  * forced split S: S ranges of whole groups per stripe.
//  * no arrival counters (more stripes than counters): one range per stripe.
int64_t gemm_mma_plan(int64_t M, int64_t N, int64_t K, int split_k, bool counters_ok, GemmArgs &g) {
    const int64_t T = (N + 15) / 16, G = groups_of(K), U = T * G;
    auto cut = [&](int64_t seglen, int64_t per, int64_t nseg) {
        g.seglen = (int)seglen, g.per = (int)per;
        g.q = (int)(seglen / per), g.rem = (int)(seglen % per);
        g.ranges = nseg * per;
    };
    if (U == 0) {
        cut(1, 1, 1);
        return 0;
    }
    if (!counters_ok || split_k == 1) {
        cut(G, 1, T);
        return 0;
    }
    if (split_k > 1) {
        const int64_t S = split_k < G ? split_k : G;
        cut(G, S, T);
        return S > 1 ? g.ranges : 0;
    }
    int64_t V = (M <= 8 ? 16 : 12) * (int64_t)W12_PLAN_SMS;
    if (V > U) V = U;
    cut(U, V, 1);
    for (int64_t v = 1; v < V; ++v) {  // any range boundary inside a stripe needs partials
        const int64_t b = v * g.q + (v < g.rem ? v : g.rem);
        if (b % G != 0) return 2 * V;
    }
    return 0;
}

cudaError_t launch_gemm_mma(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    if (g.nested8) return g.M <= 8 ? launch_nb<1, true>(t, g, s) : launch_nb<2, true>(t, g, s);
    return g.M <= 8 ? launch_nb<1, false>(t, g, s) : launch_nb<2, false>(t, g, s);
}

cudaError_t launch_gemm_mma_list(const ListParams &lp, int nb, bool nested8, int max_ctas, bool overlap,
                                 cudaStream_t s) {
    if (nested8)
        return nb == 1 ? launch_list_nb<1, true>(lp, max_ctas, overlap, s)
                       : launch_list_nb<2, true>(lp, max_ctas, overlap, s);
    return nb == 1 ? launch_list_nb<1, false>(lp, max_ctas, overlap, s)
                   : launch_list_nb<2, false>(lp, max_ctas, overlap, s);
}

}  // namespace w12
