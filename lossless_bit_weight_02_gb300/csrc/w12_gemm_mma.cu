// Small-M W12 GEMM (1 <= M <= 16): Y = A * W^T with the weights decoded in
// registers (SpecPilot, arXiv 2611.02501, section 4.1: "decodes records in
// registers", "splits the reduction in a fixed order so the GEMM is
// deterministic").
//
// Design (HBM-bound: ~1.33*M flop per weight byte):
//   * Work item = (row stripe of 16 weight rows, K-chunk s of S).  Each warp
//     streams its item's tiles: per 16x64 tile every lane issues two 128-bit
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
//   * Fixed-order reduction: chunk partials start from zero; when S > 1 they
//     go to an FP32 workspace and the last warp to finish a stripe sums them
//     in the order s = 0..S-1 and writes BF16.  S depends on (M, N, K) only,
//     so the result is identical for any grid.
#include <cstdint>

#include "w12_device.cuh"
#include "w12_internal.h"
#include "w12_stream.cuh"

namespace w12 {
namespace {

constexpr int kWarps = 4;  // warps per block; each warp keeps one 4-tile group in flight

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
    return kWarps * (4 * 32 * 16 + 2 * act_buf_bytes<NB>());
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
__device__ __forceinline__ void patch_one(uint4 (*patch)[32], uint32_t ent) {
    const int key = (int)(ent >> 16);
    const int r = (key >> 6) & 15, j = key & 63;
    const int slot = (r & 7) * 4 + (j >> 4);
    const int j16 = j & 15, pr = j16 >> 1;
    const int comp = (pr & 1) * 2 + (r >> 3);
    reinterpret_cast<uint16_t *>(&patch[pr >> 1][slot])[comp * 2 + (j16 & 1)] = (uint16_t)(ent & 0xFFFFu);
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

// One 256-column group: stage the next group's activations, then for each of
// the 4 tiles read the B fragments from shared memory, decode the two rows,
// prefetch the same tile of the next group (or, on the last group, the same
// tile again: an L2 hit), patch the tile's escapes and run the MMAs.
template <int NB>
__device__ __forceinline__ void group_step(Stream<NB> &w, const TensorView &t, const GemmArgs &g, int64_t gg,
                                           bool more, uint4 (*patch)[32], uint8_t *pw, int lane, int rows,
                                           uint32_t act, const unsigned char *actp, uint32_t frag, uint32_t c28,
                                           uint32_t c16) {
    // This lane's copies of group gg have landed; after the warp barrier so
    // have every lane's, and every lane is done reading the other buffer.
    cp_async_wait_all();
    __syncwarp();
    if (more) stage_group<NB>(act + (uint32_t)((gg + 1) & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, gg + 1, t.K, lane);
    const unsigned char *ab = actp + (gg & 1) * act_buf_bytes<NB>() + frag;
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
        decode16_fma(w.bh0[p], w.bl[p].x, w.bl[p].y, w.base2A, c28, c16, dA);
        decode16_fma(w.bh1[p], w.bl[p].z, w.bl[p].w, w.base2B, c28, c16, dB);
        w.bh0[p] = ld_stream(w.hp + next + p * 64);
        w.bh1[p] = ld_stream(w.hp + next + p * 64 + 32);
        w.bl[p] = ld_stream(w.lp + nextl + p * 32);

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
                    if (b0 + lane < w.cur.cnt && (int)(e >> 26) == p) patch_one(patch, e);
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
template <int NB>
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
        w.e_val = (uint16_t)(w.cur.ent & 0xFFFFu);
    }
}

template <int NB>  // NB = number of 8-token column blocks (1: M <= 8, 2: M <= 16)
__global__ __launch_bounds__(kWarps * 32, NB == 1 ? 4 : 3) void k_gemm_mma(TensorView t, GemmArgs g) {
    // [kWarps][4][32] uint4 escape-patch copies, then [kWarps][2][8*NB][kActPitch] activations
    extern __shared__ __align__(16) unsigned char smem[];
    uint4 (*patch)[4][32] = reinterpret_cast<uint4 (*)[4][32]>(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, q = lane & 3;
    const int S = g.split;
    const int64_t T = t.Np / 16;
    const int64_t items = T * S;
    constexpr int MP = 8 * NB;
    const uint32_t c28 = g.c28, c16 = g.c16;
    uint8_t *pw = reinterpret_cast<uint8_t *>(patch[warp]);
    const int rows = g.M < MP ? (int)g.M : MP;  // staged token rows
    // this warp's two activation buffers, and this lane's fragment in a buffer
    const unsigned char *actp = smem + kWarps * 2048 + warp * 2 * act_buf_bytes<NB>();
    const uint32_t act = (uint32_t)__cvta_generic_to_shared(actp);
    const uint32_t frag = (uint32_t)(gid * kActPitch + 16 * q) * 2u;
    grid_dep_launch();
    bool dep_done = false;

    for (int64_t item = (int64_t)blockIdx.x * kWarps + warp; item < items;
         item += (int64_t)gridDim.x * kWarps) {
        const int64_t st = item / S;
        const int s = (int)(item % S);
        // Chunk s covers whole 256-column groups [g_beg, g_end) (4 tiles each).
        const int64_t g_beg = (s * t.G) / S, g_end = ((s + 1) * t.G) / S;
        const int n0 = (int)(st * 16);  // rows < 2^30
        const int rowA = n0 + gid, rowB = n0 + gid + 8;
        Stream<NB> w;

        // 1. weight stream first, so that its latency covers the set-up below
        w.hp = reinterpret_cast<const uint4 *>(t.hi) + (st * t.KT + 4 * g_beg) * 64 + lane;
        w.lp = reinterpret_cast<const uint4 *>(t.lo) + (st * t.KT + 4 * g_beg) * 32 + lane;
        if (g_beg < g_end) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                w.bh0[p] = ld_stream(w.hp + p * 64);
                w.bh1[p] = ld_stream(w.hp + p * 64 + 32);
                w.bl[p] = ld_stream(w.lp + p * 32);
            }
        }
        // 2. bases, group offsets (lane l holds the offset of group gw0 + l),
        //    escapes of the first two groups
        w.base2A = (rowA < t.N ? (uint32_t)__ldg(t.base + rowA) : 0u) * 0x00800080u;
        w.base2B = (rowB < t.N ? (uint32_t)__ldg(t.base + rowB) : 0u) * 0x00800080u;
        const int32_t *gptr = t.esc_ptr + st * t.G;
        const int n_esc = (int)t.n_esc;  // offsets are int32
        int gw0 = (int)g_beg;
        const int gend = (int)g_end;
        auto load_window = [&](int first) -> int {
            const int gi = first + lane;
            int v = 0;
            if (gi <= gend) {
                v = __ldg(gptr + gi);
                v = v < 0 ? 0 : (v > n_esc ? n_esc : v);
            }
            return v;
        };
        int ptrw = load_window(gw0);
        auto group_bounds = [&](int gg, int &p0, int &p1) {
            if (gg + 1 - gw0 >= 32) {  // slide the window (more than 30 groups per chunk)
                gw0 = gg;
                ptrw = load_window(gw0);
            }
            p0 = __shfl_sync(kFull, ptrw, gg - gw0);
            p1 = __shfl_sync(kFull, ptrw, gg + 1 - gw0);
            if (p1 < p0) p1 = p0;
        };
        int p0 = 0, p1 = 0;
        EscBatch nxt;
        w.cur.cnt = nxt.cnt = 0;
        w.cur.ent = nxt.ent = 0;
        w.cur.p0 = nxt.p0 = 0;
        if (g_beg < g_end) {
            group_bounds((int)g_beg, p0, p1);
            w.cur = load_group_escapes(t, p0, p1, lane);
        }
        if (g_beg + 1 < g_end) {
            group_bounds((int)g_beg + 1, p0, p1);
            nxt = load_group_escapes(t, p0, p1, lane);
        }

        // Everything above reads only the W12 tensor; activations, Y and the
        // workspace may belong to the previous kernel on the stream.
        if (!dep_done) {
            grid_dep_wait();
            dep_done = true;
        }

        // Token rows beyond M are never staged: whatever their buffer rows
        // hold only reaches accumulator columns that are never stored.
#pragma unroll
        for (int b = 0; b < NB; ++b) w.acc[b][0] = w.acc[b][1] = w.acc[b][2] = w.acc[b][3] = 0.f;
        if (g_beg < g_end) {
            // every lane is done with the buffers of this warp's previous item
            __syncwarp();
            stage_group<NB>(act + (uint32_t)(g_beg & 1) * act_buf_bytes<NB>(), g.A, g.lda, rows, g_beg, t.K, lane);
            own_escape(w, lane);
        }

        for (int64_t gg = g_beg; gg < g_end; ++gg) {
            const bool more = gg + 1 < g_end;
            group_step<NB>(w, t, g, gg, more, patch[warp], pw, lane, rows, act, actp, frag, c28, c16);
            w.hp += 256;
            w.lp += 128;
            // the next group's escapes are already in flight; fetch the one after
            w.cur = nxt;
            if (more) own_escape(w, lane);
            if (gg + 2 < g_end) {
                group_bounds((int)gg + 2, p0, p1);
                nxt = load_group_escapes(t, p0, p1, lane);
            }
        }
        float (&acc)[NB][4] = w.acc;

        // Epilogue.  acc[b] = {(rowA, m0), (rowA, m0+1), (rowB, m0), (rowB, m0+1)}, m0 = 8b + 2q.
        if (S == 1) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 8 * b + 2 * q + h;
                    if (m < g.M) {
                        if (rowA < t.N) g.Y[(int64_t)m * g.ldy + rowA] = f32_to_bf16_rn(acc[b][h]);
                        if (rowB < t.N) g.Y[(int64_t)m * g.ldy + rowB] = f32_to_bf16_rn(acc[b][2 + h]);
                    }
                }
            }
        } else {
            float *P = g.partials;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                *reinterpret_cast<float2 *>(P + ((int64_t)s * t.Np + rowA) * MP + 8 * b + 2 * q) =
                    make_float2(acc[b][0], acc[b][1]);
                *reinterpret_cast<float2 *>(P + ((int64_t)s * t.Np + rowB) * MP + 8 * b + 2 * q) =
                    make_float2(acc[b][2], acc[b][3]);
            }
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = (atomicAdd(&g.counters[st], 1) == S - 1);
            last = __shfl_sync(kFull, last, 0);
            if (last) {
                __threadfence();
#pragma unroll
                for (int b = 0; b < NB; ++b) {
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int64_t row = rr ? rowB : rowA;
                        float2 v = __ldcg(reinterpret_cast<const float2 *>(P + row * MP + 8 * b + 2 * q));
                        for (int ss = 1; ss < S; ++ss) {
                            const float2 w =
                                __ldcg(reinterpret_cast<const float2 *>(P + ((int64_t)ss * t.Np + row) * MP + 8 * b + 2 * q));
                            v.x += w.x;
                            v.y += w.y;
                        }
                        if (row < t.N) {
                            const int m = 8 * b + 2 * q;
                            if (m < g.M) g.Y[(int64_t)m * g.ldy + row] = f32_to_bf16_rn(v.x);
                            if (m + 1 < g.M) g.Y[(int64_t)(m + 1) * g.ldy + row] = f32_to_bf16_rn(v.y);
                        }
                    }
                }
                if (lane == 0) g.counters[st] = 0;
            }
        }
    }
}

struct LaunchCache {
    int sms = 0;
    int occ[3] = {0, 0, 0};
};

LaunchCache &cache_for_device(int dev) {
    static LaunchCache caches[64];
    return caches[dev & 63];
}

template <int NB>
cudaError_t launch_nb(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
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
    if (lc.occ[NB] == 0) {
        int occ = 0;
        e = cudaFuncSetAttribute(k_gemm_mma<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<NB>());
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_gemm_mma<NB>, kWarps * 32, smem_bytes<NB>());
        if (e != cudaSuccess) return e;
        lc.occ[NB] = occ > 0 ? occ : 1;
    }
    const int64_t items = (t.Np / 16) * (int64_t)g.split;
    int64_t blocks = (items + kWarps - 1) / kWarps;
    const int64_t resident = (int64_t)lc.sms * lc.occ[NB];
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
    return cudaLaunchKernelEx(&cfg, k_gemm_mma<NB>, t, g);
}

}  // namespace

int64_t gemm_mma_partial_cols(int64_t M) { return M <= 8 ? 8 : 16; }

// Split factor from (M, N, K) only: as many (stripe, chunk) items as fit
// one wave of 16 resident warps on each of 152 SMs, chunks of whole
// 256-column groups.
int gemm_mma_split(int64_t M, int64_t N, int64_t K) {
    (void)M;
    const int64_t T = (N + 15) / 16, G = groups_of(K);
    if (T == 0 || G == 0) return 1;
    const int64_t target = 152 * 16;
    int64_t S = target / T;
    if (S > G) S = G;
    if (S > 32) S = 32;
    if (S < 1) S = 1;
    return (int)S;
}

cudaError_t launch_gemm_mma(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    if (g.M <= 8) return launch_nb<1>(t, g, s);
    return launch_nb<2>(t, g, s);
}

}  // namespace w12
