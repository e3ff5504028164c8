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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Copies columns 256*gg .. 256*gg+255 of the first `rows` token rows of A into
// the buffer at shared address `dst`: lane l takes columns 8l .. 8l+7 of each
// row (16 bytes; A rows are 16-byte aligned).  Columns at or beyond K read as
// zero.
template <int NB>
__device__ __forceinline__ void stage_group(uint32_t dst, const uint16_t *__restrict__ A, int64_t lda, int rows,
                                            int64_t gg, int64_t K, int lane) {
    const int64_t col = gg * 256 + 8 * lane;
    const int64_t rem = K - col;
    const uint32_t bytes = rem >= 8 ? 16u : (rem > 0 ? (uint32_t)rem * 2u : 0u);
    const uint16_t *src = bytes ? A + col : A;
    const int64_t step = bytes ? lda : 0;
#pragma unroll
    for (int i = 0; i < 8 * NB; ++i)
        if (i < rows) cp_async16(dst + (uint32_t)(i * kActPitch + 8 * lane) * 2u, src + i * step, bytes);
    cp_async_commit();
}


// Writes escape `ent` (key<<16 | bits) into the per-warp copy of the A
// fragments: slot = 4*(row%8) + col/16, component (pair&1)*2 + row/8,
// half = col&1.
__device__ __forceinline__ void patch_one(uint4 (*patch)[32], uint32_t ent, uint32_t vmask) {
    const int key = (int)(ent >> 16);
    const int r = (key >> 6) & 15, j = key & 63;
    const int slot = (r & 7) * 4 + (j >> 4);
    const int j16 = j & 15, pr = j16 >> 1;
    const int comp = (pr & 1) * 2 + (r >> 3);
    reinterpret_cast<uint16_t *>(&patch[pr >> 1][slot])[comp * 2 + (j16 & 1)] = (uint16_t)(ent & vmask);
}

// Per-warp streaming state of one work item.
template <int NB>
struct Stream {
    uint4 bh0[4], bh1[4], bl[4];  // the 4 tiles of the current group (prefetched)
    const uint4 *hp, *lp;         // hi / lo planes at the current group, this lane
    uint32_t base2A, base2B;      // row bases * 0x00800080 (rows g, g+8)
    float acc[NB][4];
    EscBatch cur;                 // escapes of the current group
    uint32_t emask;               // tiles of the group holding an escape
    uint32_t e_tile, e_off;       // this lane's escape: tile, byte in the fragment copy
    uint16_t e_val;
};

// One unit u (a 256-column group of one stripe): stage the next unit's
// activations (column group gnext), then for each of the 4 tiles read the B
// fragments from shared memory, decode the two rows, prefetch the same tile
// of the next unit (or, on the last unit, the same tile again: an L2 hit),
// patch the tile's escapes and run the MMAs.  Q: the nested 8-bit view (the
// lo plane is neither loaded nor used; escape values lose their 4 low
// mantissa bits).
template <int NB, bool Q>
__device__ __forceinline__ void group_step(Stream<NB> &w, const TensorView &t, const GemmArgs &g, int u,
                                           int gnext, bool more, uint4 (*patch)[32], uint8_t *pw, int lane,
                                           int rows, uint32_t act, const unsigned char *actp, uint32_t frag,
                                           uint32_t c28, uint32_t c16) {
    // This lane's copies for unit u have landed; after the warp barrier so
    // have every lane's, and every lane is done reading the other buffer.
    cp_async_wait_all();
    __syncwarp();
    if (more) stage_group<NB>(act + (uint32_t)((u + 1) & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, gnext, t.K, lane);
    const unsigned char *ab = actp + (u & 1) * act_buf_bytes<NB>() + frag;
    const int next = more ? 256 : 0;    // uint4 offset of the next group's hi tiles
    const int nextl = more ? 128 : 0;   // ... and lo tiles
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t bw[NB][8];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint4 *a = reinterpret_cast<const uint4 *>(ab + (8 * b * kActPitch + 64 * p) * 2);
            const uint4 v0 = a[0], v1 = a[1];
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
        w.bh0[p] = ld_stream(w.hp + next + p * 64);
        w.bh1[p] = ld_stream(w.hp + next + p * 64 + 32);
        if (!Q) w.bl[p] = ld_stream(w.lp + nextl + p * 32);

        // Escapes of this tile replace the decoded placeholders.
        if ((w.emask >> p) & 1u) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                patch[i][lane] = make_uint4(dA[2 * i], dB[2 * i], dA[2 * i + 1], dB[2 * i + 1]);
            __syncwarp();
            if (w.cur.cnt <= 32) {
                asm volatile("{\n.reg .pred pp;\nsetp.eq.u32 pp, %0, %1;\n@pp st.shared.u16 [%2], %3;\n}" ::"r"(w.e_tile),
                             "r"((uint32_t)p), "r"((uint32_t)__cvta_generic_to_shared(pw + w.e_off)), "h"(w.e_val)
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
                const uint4 v = patch[i][lane];
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
    w.e_tile = 4;
    if (lane < w.cur.cnt && w.cur.cnt <= 32) {
        const uint32_t key = w.cur.ent >> 16;
        const uint32_t r = (key >> 6) & 15, j = key & 63;
        const uint32_t slot = (r & 7) * 4 + (j >> 4), j16 = j & 15, pr = j16 >> 1;
        const uint32_t comp = (pr & 1) * 2 + (r >> 3);
        w.e_tile = key >> 10;
        w.e_off = ((pr >> 1) * 32 + slot) * 16 + comp * 4 + (j16 & 1) * 2;
        w.e_val = (uint16_t)(w.cur.ent & (Q ? 0xFFF0u : 0xFFFFu));
    }
}

template <int NB, bool Q>  // NB = number of 8-token column blocks (1: M <= 8, 2: M <= 16); Q: nested 8-bit view
__global__ __launch_bounds__(warps_of<NB>() * 32, 1) void k_gemm_mma(TensorView t, GemmArgs g) {
    constexpr int kWarps = warps_of<NB>();
    // [kWarps][4][32] uint4 escape-patch copies, then [kWarps][2][8*NB][kActPitch] activations
    extern __shared__ __align__(16) unsigned char smem[];
    uint4 (*patch)[4][32] = reinterpret_cast<uint4 (*)[4][32]>(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, q = lane & 3;
    const int G = (int)t.G;  // unit indices fit an int32 (checked on the host)
    constexpr int MP = 8 * NB;
    constexpr int kSlot = 16 * MP;  // floats in one partial (16 rows x MP tokens)
    const uint32_t c28 = g.c28, c16 = g.c16;
    uint8_t *pw = reinterpret_cast<uint8_t *>(patch[warp]);
    const int rows = g.M < MP ? (int)g.M : MP;  // staged token rows
    // this warp's two activation buffers, and this lane's fragment in a buffer
    const unsigned char *actp = smem + kWarps * 2048 + warp * 2 * act_buf_bytes<NB>();
    const uint32_t act = (uint32_t)__cvta_generic_to_shared(actp);
    const uint32_t frag = (uint32_t)(gid * kActPitch + 16 * q) * 2u;
    const uint4 *hi4 = reinterpret_cast<const uint4 *>(t.hi);
    const uint4 *lo4 = reinterpret_cast<const uint4 *>(t.lo);
    const int n_esc = (int)t.n_esc;  // offsets are int32
    grid_dep_launch();
    bool dep_done = false;

    const int ranges = (int)g.ranges;
    for (int v = blockIdx.x * kWarps + warp; v < ranges; v += gridDim.x * kWarps) {
        const int u0 = range_begin(v, g), u1 = range_begin(v + 1, g);
        if (u0 >= u1) continue;
        const int nu = (int)(u1 - u0);  // units in the range
        Stream<NB> w;

        // 1. weight stream first, so that its latency covers the set-up below
        w.hp = hi4 + (int64_t)u0 * 256 + lane;
        w.lp = lo4 + (int64_t)u0 * 128 + lane;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            w.bh0[p] = ld_stream(w.hp + p * 64);
            w.bh1[p] = ld_stream(w.hp + p * 64 + 32);
            if (!Q) w.bl[p] = ld_stream(w.lp + p * 32);
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
        // workspace may belong to the previous kernel on the stream.
        if (!dep_done) {
            grid_dep_wait();
            dep_done = true;
        }

        // every lane is done with the buffers of this warp's previous range
        __syncwarp();
        stage_group<NB>(act + (uint32_t)(u0 & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, gi, t.K, lane);
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
                group_step<NB, Q>(w, t, g, u0 + i, gi + 1 == G ? 0 : gi + 1, more, patch[warp], pw, lane, rows, act,
                               actp, frag, c28, c16);
                w.hp += 256;
                w.lp += 128;
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
                            if (rowA < t.N) g.Y[(int64_t)m * g.ldy + rowA] = f32_to_bf16_rn(w.acc[b][h]);
                            if (rowB < t.N) g.Y[(int64_t)m * g.ldy + rowB] = f32_to_bf16_rn(w.acc[b][2 + h]);
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
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int lr = gid + 8 * rr;
                    const int off = lr * MP + 8 * b + 2 * q;
                    float2 sum = __ldcg(reinterpret_cast<const float2 *>(first + off));
                    for (int x = va + 1; x <= vb; x += 4) {  // four independent loads at a time
                        float2 y[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (x + j <= vb)
                                y[j] = __ldcg(reinterpret_cast<const float2 *>(g.partials + (int64_t)(x + j) * kSlot + off));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (x + j <= vb) {
                                sum.x += y[j].x;
                                sum.y += y[j].y;
                            }
                    }
                    const int row = rs * 16 + lr;
                    if (row < t.N) {
                        const int m = 8 * b + 2 * q;
                        if (m < g.M) g.Y[(int64_t)m * g.ldy + row] = f32_to_bf16_rn(sum.x);
                        if (m + 1 < g.M) g.Y[(int64_t)(m + 1) * g.ldy + row] = f32_to_bf16_rn(sum.y);
                    }
                }
            }
            if (lane == 0) g.counters[rs] = 0;
        }
    }
}

struct LaunchCache {
    int sms = 0;
    int occ[3][2] = {};
};

LaunchCache &cache_for_device(int dev) {
    static LaunchCache caches[64];
    return caches[dev & 63];
}

template <int NB, bool Q>
cudaError_t launch_nb(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    constexpr int kWarps = warps_of<NB>();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    LaunchCache &lc = cache_for_device(dev);
    if (lc.sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        lc.sms = sms;
    }
    int &occ_slot = lc.occ[NB][Q ? 1 : 0];
    if (occ_slot == 0) {
        int occ = 0;
        e = cudaFuncSetAttribute(k_gemm_mma<NB, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<NB>());
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_gemm_mma<NB, Q>, kWarps * 32, smem_bytes<NB>());
        if (e != cudaSuccess) return e;
        occ_slot = occ > 0 ? occ : 1;
    }
    int64_t blocks = (g.ranges + kWarps - 1) / kWarps;
    const int64_t resident = (int64_t)lc.sms * occ_slot;
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

}  // namespace w12
