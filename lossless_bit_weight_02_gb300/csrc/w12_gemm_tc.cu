// W12 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM) for
// 16 <= Mpad <= 256 tokens: Y = A * W^T with W decoded on the fly
// (SpecPilot, arXiv 2611.02501, section 4.1: the GEMM decodes the records in
// registers and splits its reduction in a fixed order).
//
// One CTA owns 128 weight rows (8 stripes of 16) and a chunk of whole
// 256-column groups.  Two builds of the kernel: one CTA per SM with 16
// decoder warps (two per stripe), or two CTAs per SM with 8 decoder warps
// (one per stripe) each; the second wins when the grid holds enough CTAs to
// fill 2 x 152 slots.  Per 64-column k-block:
//   * a weight-producer warp fetches the 8 tiles of the k-block (12 KB of
//     W12 planes) with two tiled TMA copies (the planes seen as 4-D u8
//     tensors), up to a whole ring of k-blocks ahead of the decoders;
//   * the decoder warps (one or two per stripe, taking every k-block, or
//     the even / odd ones) read their
//     tile from that ring (the fragment-native order makes this three
//     conflict-free 16-byte loads per lane), decode it in registers and
//     store it as BF16 into the UMMA A operand: 128 rows x 128 bytes,
//     K-major, 128-byte swizzle.  Escapes of the tile are written over
//     their slots.  Each warp then fences the generic->async proxy and one
//     lane arrives on the stage's "A full" barrier;
//   * an activation-producer warp loads the tile [Mpad x 64] with TMA (rows
//     >= M and columns >= K come back as zeros) into the B operand;
//   * an MMA warp waits for both, and one elected lane issues four
//     tcgen05.mma (M=128, N=Mpad, K=16) accumulating in TMEM and commits to
//     the stages' "empty" barriers.  The producer and MMA loops run on the
//     whole (converged) warp so that their addresses stay in uniform
//     registers; only the issue is elected.
// Ring depths (decoded A, weight planes, activations) fill the shared
// memory for the given Mpad.  The epilogue warps read the accumulator with
// tcgen05.ld.  With a split of S > 1 the chunk partials go to the FP32
// workspace and the last CTA of a row tile adds them in the order
// s = 0..S-1; S depends only on (M, N, K).  The work items (row tile,
// K-chunk) or balanced ranges are fixed by (M, N, K) too; a CTA walks items
// blockIdx.x, blockIdx.x + gridDim.x, ..., so a grid capped by
// w12_gemm_opts.max_ctas computes bitwise the same result.
// Every mbarrier wait is bounded in time (about a second, read from the
// global nanosecond timer): on expiry the CTA records W12_ERR_TIMEOUT in the
// workspace error word, waits (bounded) for its own copies and MMAs, and
// frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "w12_device.cuh"
#include "w12_internal.h"
#include "w12_stream.cuh"

namespace w12 {
namespace {

// Warp roles of a CTA with D decoder warps (D = 16: two per 16-row stripe,
// even / odd k-blocks, one CTA per SM; D = 8: one per stripe, two CTAs per
// SM): warps 0..D-1 decode, D streams the weight planes (and owns TMEM),
// D+1 streams the activations, D+2 issues the MMAs.
template <int D>
struct Roles {
    static constexpr int kDecWarps = D;
    static constexpr int kPar = D / 8;          // decoder warps per stripe
    static constexpr int kCtasPerSm = 16 / D;
    static constexpr int kWProdWarp = D;
    static constexpr int kBProdWarp = D + 1;
    static constexpr int kMmaWarp = D + 2;
    static constexpr int kThreads = 32 * (D + 3);
};
constexpr uint32_t kAStageBytes = 128 * 128;   // decoded A: 128 rows x 64 BF16, swizzled
constexpr uint32_t kWStageBytes = 8 * 1536;    // the 8 stripes of a row tile, one k-block: 8 KB hi, 4 KB lo
constexpr int kMaxStages = 12;   // per ring
constexpr uint64_t kWaitNs = 1000000000ull;    // a wait gives up after ~1 s ...
constexpr long long kWaitPollCap = 1LL << 28;  // ... or after this many polls, whichever comes first
// A grid of at least this many CTAs takes the two-CTAs-per-SM build (about
// 85% of its 2 x 152 slots); measured on GB300, smaller grids ran faster with
// 16 decoder warps per CTA.
constexpr int64_t kTwoPerSmMinCtas = 258;

struct TcParams {
    int Mp;                // tokens padded to a multiple of 16 (UMMA N)
    int a_st, w_st, b_st;  // depths of the decoded-A, weight-plane and activation rings (2..kMaxStages)
    int tmem_cols;         // power of two >= max(32, Mp)
    uint32_t idesc;        // tcgen05 instruction descriptor
};

// Stage index and phase parity of a ring position, advanced by `step`
// positions at a time (step <= depth).
struct RingPos {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int step, int depth) {
        stage += step;
        if (stage >= depth) {
            stage -= depth;
            phase ^= 1u;
        }
    }
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// try_wait without a time hint: returns when the phase completes or after
// a short, hardware-chosen time.  (A suspend-time hint made every wait a few
// percent slower on GB300: the thread wakes later after the phase flips.)
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the completion of phase `parity`.  Gives up (returns
// false) when another thread of the CTA has given up, or after kWaitNs (or
// kWaitPollCap polls), in which case it raises the CTA's abort flag and the
// error word.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (long long i = 1; i < kWaitPollCap; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitNs) break;
        }
    }
    *abort_flag = 1;
    atomicExch(err, 1);
    return false;
}

// Bounded wait that does not give up when the CTA aborts: for work already
// handed to the asynchronous units (TMA copies, MMAs), which must finish
// before the CTA may free its shared memory and TMEM.  Returns false (and
// raises the error word) only when the limit runs out.
__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity, int32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (long long i = 1; i < kWaitPollCap; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0 && global_ns() - t0 > kWaitNs) break;
    }
    atomicExch(err, 1);
    return false;
}

// true on one lane of the (converged) warp
__device__ __forceinline__ bool elect_one() {
    uint32_t r;
    asm volatile("{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}" : "=r"(r));
    return r != 0;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand with 128-byte swizzle: 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu)   // start address
           | ((uint64_t)1 << 16)                // leading byte offset (unused for swizzled K-major)
           | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows x 128 B
           | ((uint64_t)1 << 46)                // descriptor version
           | ((uint64_t)2 << 61);               // swizzle: 128 bytes
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Fetch a tensor map (a __grid_constant__ kernel parameter) ahead of its first copy.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Thread-block clusters (the split-K CTAs of one row tile): rank in the
// cluster, a cluster-wide barrier (every thread of every CTA), and 16-byte
// loads from another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cluster4(uint32_t local_addr, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// Byte offset of (row r, 16-byte chunk c) in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c2, int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(c2), "r"(c3), "r"(smem_addr(bar))
        : "memory");
}

// tmap: activations [M, K] BF16, box [Mp, 64], 128-byte swizzle.
// hmap / lmap: the hi / lo plane as u8 [stripes][k-blocks][4 or 2][256], box
// [8 stripes][1 k-block][4 or 2][256]: one copy brings the row tile's 8
// tiles of a k-block (stripes past the end read as zero).
//
// Work items are (row tile, K-chunk) pairs, item = row_tile*S + chunk.  A CTA
// takes items blockIdx.x, blockIdx.x + gridDim.x, ...: with the default grid
// (one CTA per item) that is one item, with a capped grid several.  The rings
// and their phases run on from one item to the next; the accumulator in TMEM
// is reused, and every decoder warp finishes reading it (the item's epilogue)
// before any of them decodes a tile of the next item, so no MMA of the next
// item can overwrite it early.  The item, its chunk bounds and the order of
// the split-K sum depend on (M, N, K) only, never on the grid.
template <int D, bool SILU, bool PERSIST, bool CLUSTER>
__global__ __launch_bounds__(Roles<D>::kThreads, Roles<D>::kCtasPerSm) void k_gemm_tc(
    TensorView t, GemmArgs g, TcParams tp, const __grid_constant__ CUtensorMap tmap,
    const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap lmap) {
    using R = Roles<D>;
    constexpr int kDecWarps = R::kDecWarps, kPar = R::kPar;
    constexpr int kWProdWarp = R::kWProdWarp, kBProdWarp = R::kBProdWarp, kMmaWarp = R::kMmaWarp;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned, by an offset so that the compiler keeps the
    // shared address space (ld.shared / st.shared, not generic accesses)
    uint8_t *base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int RA = tp.a_st, RW = tp.w_st, RB = tp.b_st, Mp = tp.Mp;
    const uint32_t b_stage_bytes = (uint32_t)Mp * 128;
    uint8_t *a_st = base;                                // RA x 16 KB (1024-aligned)
    uint8_t *b_st = a_st + RA * kAStageBytes;            // RB x Mp*128 B (1024-aligned)
    uint8_t *w_st = b_st + RB * b_stage_bytes;           // RW x 12 KB (1024-aligned)
    uint64_t *w_full = reinterpret_cast<uint64_t *>(w_st + RW * kWStageBytes);
    uint64_t *w_empty = w_full + RW;
    uint64_t *a_full = w_empty + RW;
    uint64_t *a_empty = a_full + RA;
    uint64_t *b_full = a_empty + RA;
    uint64_t *b_empty = b_full + RB;
    uint64_t *done = b_empty + RB;  // one phase per item: its MMAs have completed
    uint64_t *fin = done + 1;        // the MMA warp's own last wait: every MMA it issued has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = g.split;
    const int64_t T = t.Np / 16;
    const int items = (int)((t.Np + 127) / 128) * S;
    // Without PERSIST the grid holds one CTA per item, and a stride of
    // `items` lets the compiler see that every loop below runs once (the
    // loop over items, kept general, made the kernel ~9% slower on GB300).
    const int stride = PERSIST ? (int)gridDim.x : items;
    // groups [g_beg, g_end) of item `item` and its row tile
    auto item_span = [&](int item, int64_t &tt, int64_t &g_beg, int64_t &g_end) {
        tt = item / S;
        const int s = item - (int)tt * S;
        g_beg = (s * t.G) / S;
        g_end = ((s + 1) * t.G) / S;
    };

    // The first item starts at once, while the other barriers and TMEM are
    // set up: the decoders load its bases and group offsets (kept raw until
    // after the setup barrier, so no warp waits for them there; the escape
    // entries, which need the offsets, follow in the item loop), and the
    // weight producer initialises its own ring's barriers and issues the
    // first ring-full of plane copies.  Both read only the W12 tensor.
    int pre_ptrw = 0;
    uint32_t pre_bA = 0, pre_bB = 0;
    if (warp < kDecWarps && (int)blockIdx.x < items) {
        int64_t tt0, gb0, ge0;
        item_span((int)blockIdx.x, tt0, gb0, ge0);
        const int64_t st0 = tt0 * 8 + (warp & 7);
        if (st0 < T && ge0 > gb0) {
            const int gi = (int)gb0 + lane;
            if (gi <= (int)ge0) pre_ptrw = __ldg(t.esc_ptr + st0 * t.G + gi);
            const int64_t nA = st0 * 16 + (lane >> 2), nB = nA + 8;
            if (nA < t.N) pre_bA = __ldg(t.base + nA);
            if (nB < t.N) pre_bB = __ldg(t.base + nB);
        }
    }
    int pre_issued = 0;  // plane copies of the first item already in flight
    if (warp == kWProdWarp) {
        if (lane == 0) {
            prefetch_tmap(&hmap);
            if (!g.nested8) prefetch_tmap(&lmap);
            for (int i = 0; i < RW; ++i) {
                mbar_init(&w_full[i], 1);    // the producer's expect_tx
                mbar_init(&w_empty[i], 8);   // one arrival per stripe's decoder warp of the k-block
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        if ((int)blockIdx.x < items) {
            int64_t tt0, gb0, ge0;
            item_span((int)blockIdx.x, tt0, gb0, ge0);
            const int nkb0 = (int)(4 * (ge0 - gb0));
            pre_issued = nkb0 < RW ? nkb0 : RW;
            if (lane == 0) {  // the ring is empty: no slot to wait for
                for (int kb = 0; kb < pre_issued; ++kb) {
                    mbar_expect_tx(&w_full[kb], g.nested8 ? 8192u : kWStageBytes);
                    uint8_t *dst = w_st + kb * kWStageBytes;
                    tma_load_4d(dst, &hmap, (int)(4 * gb0) + kb, (int)(tt0 * 8), &w_full[kb]);
                    if (!g.nested8) tma_load_4d(dst + 8192, &lmap, (int)(4 * gb0) + kb, (int)(tt0 * 8), &w_full[kb]);
                }
            }
        }
        __syncwarp();
    } else if (warp == kBProdWarp && lane == 0) {
        prefetch_tmap(&tmap);
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < RA; ++i) {
            mbar_init(&a_full[i], 8);
            mbar_init(&a_empty[i], 1);               // tcgen05.commit
        }
        for (int i = 0; i < RB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        mbar_init(done, 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWProdWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(tp.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch();

    if (warp < kDecWarps) {
        // ------------------------------------------------------------------
        // Decoders: warp w handles stripe st = 8*tt + (w%8) on every k-block
        // (8 decoder warps) or on the k-blocks of parity w/8 (16 warps:
        // tiles p = w/8 and w/8 + 2 of every group): the tile's planes come
        // from the weight ring, the BF16 tile goes to the A ring (K-major,
        // 128-byte swizzle), escapes over their slots.  Every decoder warp
        // runs every item and every named barrier, also after an abort
        // (its waits then return at once), so the barriers always match.
        // ------------------------------------------------------------------
        const int gid = lane >> 2, q = lane & 3;
        const int sw = warp & 7, par = warp >> 3;
        const int rA = 16 * sw + gid, rB = rA + 8;
        const uint32_t c28 = g.c28, c16 = g.c16;
        const uint32_t vmask = g.nested8 ? 0xFFF0u : 0xFFFFu;  // escape bits kept
        const int n_esc = (int)t.n_esc;
        const int quarter = warp & 3, half = warp >> 2;  // epilogue: TMEM lanes 32*quarter..; half: 0 .. kDecWarps/4 - 1
        const int chunks = Mp / 16;
        RingPos wp, ap;   // ring positions of this warp's next k-block
        wp.advance(par, RW);
        ap.advance(par, RA);
        int it = 0;  // items this CTA has done
        for (int item = blockIdx.x; item < items; item += stride, ++it) {
            int64_t tt, g_beg, g_end;
            item_span(item, tt, g_beg, g_end);
            const int nkb = (int)(4 * (g_end - g_beg));
            const int64_t st = tt * 8 + sw;
            const bool live = st < T;  // warp-uniform
            uint32_t base2A = 0, base2B = 0;
            EscBatch cur, nxt;
            cur.cnt = nxt.cnt = 0;
            cur.ent = nxt.ent = 0;
            cur.p0 = nxt.p0 = 0;
            const int32_t *gptr = t.esc_ptr + (live ? st : 0) * t.G;
            // group offsets: lane l holds the offset of group gw0 + l (one
            // coalesced load per 31 groups, no dependent load inside the loop)
            int gw0 = (int)g_beg;
            const int gend = (int)g_end;
            auto load_window = [&](int first) -> int {
                const int gi = first + lane;
                int v = 0;
                if (live && gi <= gend) {
                    v = __ldg(gptr + gi);
                    v = v < 0 ? 0 : (v > n_esc ? n_esc : v);
                }
                return v;
            };
            int ptrw = it == 0 ? (pre_ptrw < 0 ? 0 : (pre_ptrw > n_esc ? n_esc : pre_ptrw)) : load_window(gw0);
            auto bounds = [&](int64_t gg64, int &p0, int &p1) {
                const int gg = (int)gg64;
                if (gg + 1 - gw0 >= 32) {  // slide the window (more than 30 groups per chunk)
                    gw0 = gg;
                    ptrw = load_window(gw0);
                }
                p0 = __shfl_sync(kFull, ptrw, gg - gw0);
                p1 = __shfl_sync(kFull, ptrw, gg + 1 - gw0);
                if (p1 < p0) p1 = p0;
            };
            if (live && nkb > 0) {
                if (it == 0) {
                    base2A = pre_bA * 0x00800080u;
                    base2B = pre_bB * 0x00800080u;
                } else {
                    const int64_t nA = st * 16 + gid, nB = nA + 8;
                    base2A = (nA < t.N ? (uint32_t)__ldg(t.base + nA) : 0u) * 0x00800080u;
                    base2B = (nB < t.N ? (uint32_t)__ldg(t.base + nB) : 0u) * 0x00800080u;
                }
                int p0, p1;
                bounds(g_beg, p0, p1);
                cur = load_group_escapes(t, p0, p1, lane);
                if (g_beg + 1 < g_end) {
                    bounds(g_beg + 1, p0, p1);
                    nxt = load_group_escapes(t, p0, p1, lane);
                }
            }
            uint32_t emask = (live && nkb > 0) ? escape_tiles(cur, lane) : 0u;
            // Y and the workspace may belong to the previous kernel (the
            // first item's metadata above reads only the W12 tensor)
            if (it == 0) grid_dep_wait();
            bool ok = !*abort_flag;
            for (int kb = par; kb < nkb && ok; kb += kPar, wp.advance(kPar, RW), ap.advance(kPar, RA)) {
                const int p = kb & 3;  // tile of the group
                if (kb >= 4 && p == par && live) {  // first tile of a new group for this warp
                    const int64_t gg = g_beg + (kb >> 2);
                    cur = nxt;
                    emask = escape_tiles(cur, lane);
                    if (gg + 1 < g_end) {
                        int p0, p1;
                        bounds(gg + 1, p0, p1);
                        nxt = load_group_escapes(t, p0, p1, lane);
                    }
                }
                const int ws = wp.stage, as = ap.stage;
                const uint32_t wph = wp.phase, aph = ap.phase;
                // the whole warp leaves together, so no lane is left behind at a
                // warp-wide instruction
                if (!__all_sync(kFull, mbar_wait(&w_full[ws], wph, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                uint32_t dA[8], dB[8];
                if (live) {
                    const uint8_t *W = w_st + ws * kWStageBytes;
                    const uint4 h0 = lds128(W + sw * 1024 + lane * 16), h1 = lds128(W + sw * 1024 + 512 + lane * 16);
                    // the nested 8-bit view reads no lo plane: records with zero low nibbles
                    const uint4 l = g.nested8 ? make_uint4(0u, 0u, 0u, 0u) : lds128(W + 8192 + sw * 512 + lane * 16);
                    decode16_fma(h0, l.x, l.y, base2A, c28, c16, dA);
                    decode16_fma(h1, l.z, l.w, base2B, c28, c16, dB);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);  // the planes are in registers
                if (!__all_sync(kFull, mbar_wait(&a_empty[as], aph ^ 1u, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                if (live) {
                    uint8_t *A = a_st + as * kAStageBytes;
                    *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q)) = make_uint4(dA[0], dA[1], dA[2], dA[3]);
                    *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q + 1)) = make_uint4(dA[4], dA[5], dA[6], dA[7]);
                    *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q)) = make_uint4(dB[0], dB[1], dB[2], dB[3]);
                    *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q + 1)) = make_uint4(dB[4], dB[5], dB[6], dB[7]);
                    if ((emask >> p) & 1u) {  // escapes of this tile overwrite their slots
                        __syncwarp();
                        auto put = [&](uint32_t e) {
                            const int key = (int)(e >> 16);
                            const int r = 16 * sw + ((key >> 6) & 15), j = key & 63;
                            *reinterpret_cast<uint16_t *>(A + swz(r, j >> 3) + (j & 7) * 2) = (uint16_t)(e & vmask);
                        };
                        if (cur.cnt <= 32) {
                            if (lane < cur.cnt && (int)(cur.ent >> 26) == p) put(cur.ent);
                        } else {
                            for (int b0 = 0; b0 < cur.cnt; b0 += 32) {
                                const uint32_t e = (b0 + lane < cur.cnt) ? __ldg(t.esc + cur.p0 + b0 + lane) : 0u;
                                if (b0 + lane < cur.cnt && (int)(e >> 26) == p) put(e);
                            }
                        }
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[as]);
            }

            // --------------------------------------------------------------
            // Epilogue: TMEM lanes 32*(warp%4).. ; the warps w, w+4, ... (two
            // or four of them) split the 16-column chunks.
            // --------------------------------------------------------------
            // every MMA of the item has completed (a wait that gives up on an
            // abort: the MMA warp then no longer keeps pace with the items,
            // and it waits for its own MMAs before the CTA exits)
            const bool mma_done = __all_sync(kFull, mbar_wait(done, (uint32_t)(it & 1), abort_flag, g.error));
            tc_fence_after();
            const int64_t n = tt * 128 + 32 * quarter + lane;
            const int s = item - (int)tt * S;
            const bool have = __all_sync(kFull, mma_done && ok && !*abort_flag);
            if (have) {
                for (int c = half; c < chunks; c += kDecWarps / 4) {
                    float v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(16 * c), v);
                    if (SILU && S == 1) {  // hidden unit 8*(n/16) + n%16 on the gate lanes
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float y = silu_pair(v[j]);
                            const int m = 16 * c + j;
                            if (!(lane & 8) && n < t.N && m < g.M)
                                g.Y[(int64_t)m * g.ldy + (n >> 4) * 8 + (n & 7)] = f32_to_bf16_rn(y);
                        }
                    } else if (S == 1) {
                        if (n < t.N) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int m = 16 * c + j;
                                if (m < g.M) g.Y[(int64_t)m * g.ldy + n] = f32_to_bf16_rn(v[j]);
                            }
                        }
                    } else if (CLUSTER) {  // the CTA's partial [m][128 rows] in its own shared memory
                        float *part = reinterpret_cast<float *>(base);
#pragma unroll
                        for (int j = 0; j < 16; ++j) part[(16 * c + j) * 128 + 32 * quarter + lane] = v[j];
                    } else if (n < t.Np) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            g.partials[((int64_t)s * Mp + 16 * c + j) * t.Np + n] = v[j];
                    }
                }
            }
            // every decoder warp is done reading the accumulator before any of
            // them hands the MMA warp a tile of the next item
            tc_fence_before();
            if (S > 1 && !CLUSTER) __threadfence();
            asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
            if (S > 1 && !CLUSTER) {
                // fixed-order combination by the last CTA of this row tile
                if (threadIdx.x == 0) *last_flag = have ? (atomicAdd(&g.counters[tt], 1) == S - 1) : 0;
                asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
                if (*last_flag && SILU) {
                    __threadfence();
                    const bool valid = n < t.N;  // the same for a gate lane and its up lane (N % 16 == 0)
                    for (int c = half; c < chunks; c += kDecWarps / 4) {
                        float acc[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                        if (valid) {
                            for (int ss = 0; ss < S; ++ss) {  // in the order s = 0..S-1
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    acc[j] += __ldcg(g.partials + ((int64_t)ss * Mp + 16 * c + j) * t.Np + n);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float y = silu_pair(acc[j]);
                            if (!(lane & 8) && valid && 16 * c + j < g.M)
                                g.Y[(int64_t)(16 * c + j) * g.ldy + (n >> 4) * 8 + (n & 7)] = f32_to_bf16_rn(y);
                        }
                    }
                } else if (*last_flag) {
                    __threadfence();
                    if (n < t.N) {
                        auto part = [&](int ss, int c, int j) {
                            return __ldcg(g.partials + ((int64_t)ss * Mp + 16 * c + j) * t.Np + n);
                        };
                        for (int c = half; c < chunks; c += kDecWarps / 4) {
                            // summed in the order s = 0..S-1; the loads of four
                            // chunks at a time are in flight together
                            float acc[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] = part(0, c, j);
                            int ss = 1;
                            for (; ss + 3 < S; ss += 4) {
                                float v[4][16];
#pragma unroll
                                for (int b = 0; b < 4; ++b)
#pragma unroll
                                    for (int j = 0; j < 16; ++j) v[b][j] = part(ss + b, c, j);
#pragma unroll
                                for (int b = 0; b < 4; ++b)
#pragma unroll
                                    for (int j = 0; j < 16; ++j) acc[j] += v[b][j];
                            }
                            for (; ss < S; ++ss) {
                                float v[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[j] = part(ss, c, j);
#pragma unroll
                                for (int j = 0; j < 16; ++j) acc[j] += v[j];
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (16 * c + j < g.M) g.Y[(int64_t)(16 * c + j) * g.ldy + n] = f32_to_bf16_rn(acc[j]);
                        }
                    }
                }
                if (*last_flag && threadIdx.x == 0) g.counters[tt] = 0;
                // (thread 0 writes last_flag again only after the next item's
                // first barrier, which every decoder warp reaches after
                // reading it here)
            }
        }
    } else if (warp == kWProdWarp) {
        // ------------------------------------------------------------------
        // Weight planes: one k-block (8 tiles of 1.5 KB) per stage, with
        // tiled copies, up to RW k-blocks ahead of the decoders, item after
        // item.  Reads only the W12 tensor, so it starts before the previous
        // kernel ends.
        // ------------------------------------------------------------------
        // The whole warp runs the loop (warp-uniform values stay in uniform
        // registers); one elected lane issues.
        int issued = 0;
        bool ok = true;
        RingPos wp;
        for (int item = blockIdx.x; item < items && ok; item += stride) {
            int64_t tt, g_beg, g_end;
            item_span(item, tt, g_beg, g_end);
            const int nkb = (int)(4 * (g_end - g_beg));
            for (int kb = 0; kb < nkb; ++kb, wp.advance(1, RW)) {
                if (item == (int)blockIdx.x && kb < pre_issued) {  // issued before the setup barrier
                    ++issued;
                    continue;
                }
                const int ws = wp.stage;
                if (!__all_sync(kFull, mbar_wait(&w_empty[ws], wp.phase ^ 1u, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    // the full box is counted, out-of-range stripes included (zero-filled)
                    mbar_expect_tx(&w_full[ws], g.nested8 ? 8192u : kWStageBytes);
                    uint8_t *dst = w_st + ws * kWStageBytes;
                    const int kbg = (int)(4 * g_beg) + kb, st0 = (int)(tt * 8);
                    tma_load_4d(dst, &hmap, kbg, st0, &w_full[ws]);
                    if (!g.nested8) tma_load_4d(dst + 8192, &lmap, kbg, st0, &w_full[ws]);
                }
                __syncwarp();
                ++issued;
            }
        }
        // the copies issued last must have landed before the CTA exits
        for (int i = issued > RW ? issued - RW : 0; i < issued; ++i)
            mbar_drain(&w_full[i % RW], (uint32_t)((i / RW) & 1), g.error);
    } else if (warp == kBProdWarp) {
        // ------------------------------------------------------------------
        // Activations: one TMA tile [Mp x 64] per k-block.
        // ------------------------------------------------------------------
        grid_dep_wait();  // A may be written by the previous kernel
        int issued = 0;
        bool ok = true;
        RingPos bp;
        for (int item = blockIdx.x; item < items && ok; item += stride) {
            int64_t tt, g_beg, g_end;
            item_span(item, tt, g_beg, g_end);
            const int nkb = (int)(4 * (g_end - g_beg));
            for (int kb = 0; kb < nkb; ++kb, bp.advance(1, RB)) {
                const int stage = bp.stage;
                if (!__all_sync(kFull, mbar_wait(&b_empty[stage], bp.phase ^ 1u, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    mbar_expect_tx(&b_full[stage], b_stage_bytes);
                    tma_load_2d(b_st + stage * b_stage_bytes, &tmap, (int)((4 * g_beg + kb) * 64), 0,
                                &b_full[stage]);
                }
                __syncwarp();
                ++issued;
            }
        }
        // the copies issued last must have landed before the CTA exits
        for (int i = issued > RB ? issued - RB : 0; i < issued; ++i)
            mbar_drain(&b_full[i % RB], (uint32_t)((i / RB) & 1), g.error);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------
        // MMA issue.  After each item's MMAs (or, after an abort, none) a
        // commit completes that item's phase of `done`, so the decoders'
        // epilogue never waits longer than the MMAs already issued.
        // ------------------------------------------------------------------
        // The whole warp runs the loop; one elected lane issues the MMAs.
        if (g.test_stall)  // a wait that nothing completes: it runs out and aborts the CTA
            (void)__all_sync(kFull, mbar_wait(fin, 0, abort_flag, g.error));
        RingPos ap, bp;
        bool ok = true;
        for (int item = blockIdx.x; item < items; item += stride) {
            int64_t tt, g_beg, g_end;
            item_span(item, tt, g_beg, g_end);
            const int nkb = (int)(4 * (g_end - g_beg));
            for (int kb = 0; kb < nkb && ok; ++kb, ap.advance(1, RA), bp.advance(1, RB)) {
                const int as = ap.stage, bs = bp.stage;
                if (!__all_sync(kFull, mbar_wait(&a_full[as], ap.phase, abort_flag, g.error)) ||
                    !__all_sync(kFull, mbar_wait(&b_full[bs], bp.phase, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(a_st + as * kAStageBytes);
                const uint32_t b0 = smem_addr(b_st + bs * b_stage_bytes);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma(tmem, smem_desc(a0 + 32 * kk), smem_desc(b0 + 32 * kk), tp.idesc, (kb | kk) != 0);
                    umma_commit(&a_empty[as]);
                    umma_commit(&b_empty[bs]);
                }
                __syncwarp();
            }
            if (elect_one()) umma_commit(done);  // arrives once every MMA issued above has completed
            __syncwarp();
        }
        // TMEM and the shared-memory operands stay allocated until every MMA
        // issued has completed (after an abort the decoders stop waiting)
        if (elect_one()) umma_commit(fin);
        __syncwarp();
        (void)__all_sync(kFull, mbar_drain(fin, 0, g.error));
    }

    tc_fence_before();
    __syncthreads();
    if (CLUSTER) {
        // The S CTAs of row tile tt form one cluster (rank = chunk s).  Each
        // has its FP32 partial [m][128] in its own shared memory; after the
        // barrier the cluster combines them, CTA r taking the rows m = r,
        // r + S, ...: every output is summed over s = 0..S-1 in that order,
        // exactly as the global-memory path does.
        cluster_sync();
        if (warp < kDecWarps) {
            const int r = (int)cluster_ctarank();
            const int64_t tt = (int64_t)blockIdx.x / S;
            const int qd = threadIdx.x & 31, rs = threadIdx.x >> 5;
            const int64_t n0 = tt * 128 + 4 * qd;  // this thread's 4 weight rows
            const uint32_t local = smem_addr(base) + (uint32_t)qd * 16u;
            const int mmax = Mp < (int)g.M ? Mp : (int)g.M;
            for (int m = r + S * rs; m < mmax; m += S * kDecWarps) {
                const uint32_t row = local + (uint32_t)m * 512u;
                if (!SILU) {
                    if (n0 >= t.N) continue;
                    float4 p[8];
#pragma unroll
                    for (int ss = 0; ss < 8; ++ss)
                        if (ss < S) p[ss] = ld_cluster4(row, (uint32_t)ss);
                    float4 acc = p[0];
#pragma unroll
                    for (int ss = 1; ss < 8; ++ss) {
                        if (ss < S) {
                            acc.x += p[ss].x;
                            acc.y += p[ss].y;
                            acc.z += p[ss].z;
                            acc.w += p[ss].w;
                        }
                    }
                    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (n0 + i < t.N) g.Y[(int64_t)m * g.ldy + n0 + i] = f32_to_bf16_rn(a[i]);
                } else {
                    // gate rows 16h..16h+7, up rows 16h+8..16h+15: a gate quad
                    // takes its up quad 8 rows on (N % 16 == 0)
                    if ((qd & 2) || n0 >= t.N) continue;
                    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // gate rows, then up rows
                        float4 pp[8];
#pragma unroll
                        for (int ss = 0; ss < 8; ++ss)
                            if (ss < S) pp[ss] = ld_cluster4(row + 32u * h, (uint32_t)ss);
                        float *a = h ? au : ag;
#pragma unroll
                        for (int ss = 0; ss < 8; ++ss)
                            if (ss < S) a[0] += pp[ss].x, a[1] += pp[ss].y, a[2] += pp[ss].z, a[3] += pp[ss].w;
                    }
                    const int64_t col = (n0 >> 4) * 8 + (n0 & 15);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        g.Y[(int64_t)m * g.ldy + col + i] = f32_to_bf16_rn(silu_f32(ag[i]) * au[i]);
                }
            }
        }
        cluster_sync();  // no CTA leaves while another still reads its partial
    }
    if (warp == kWProdWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tp.tmem_cols)
                     : "memory");
    }
}

// Balanced range cut (used for Mpad > 128 on large layers, one CTA per SM):
// the units u = row_tile*G + group are cut into V contiguous ranges
// (range_begin), one per SM-sized share, so every SM streams the same number
// of units whatever the row-tile count.  A CTA takes ranges blockIdx.x,
// blockIdx.x + gridDim.x, ... (one with the default grid of V CTAs).  A range
// is walked piece by piece (the part of it inside one row tile).  The CTA's
// pieces, counted over all its ranges, alternate between two TMEM
// accumulator buffers; a piece's epilogue is deferred until the piece two
// later needs its buffer (for most ranges, to the range's end), so the
// decoders go straight on to the next row tile, whose bases and group offsets
// they fetch during the last group of the current one.  A piece that covers
// its whole row tile is rounded and stored; the range's first and last
// pieces otherwise go to FP32 slots v and v + V, and the last CTA to arrive
// at a row tile sums its pieces in range order.  The ranges and the order of
// every sum depend on (M, N, K) only, never on the grid.
template <int D, bool SILU, bool PERSIST>
__global__ __launch_bounds__(Roles<D>::kThreads, Roles<D>::kCtasPerSm) void k_gemm_tc_ranges(
    TensorView t, GemmArgs g, TcParams tp, const __grid_constant__ CUtensorMap tmap,
    const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap lmap) {
    using R = Roles<D>;
    constexpr int kDecWarps = R::kDecWarps, kPar = R::kPar;
    constexpr int kWProdWarp = R::kWProdWarp, kBProdWarp = R::kBProdWarp, kMmaWarp = R::kMmaWarp;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned, by an offset so that the compiler keeps the
    // shared address space (ld.shared / st.shared, not generic accesses)
    uint8_t *base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int RA = tp.a_st, RW = tp.w_st, RB = tp.b_st, Mp = tp.Mp;
    const uint32_t b_stage_bytes = (uint32_t)Mp * 128;
    uint8_t *a_st = base;                                // RA x 16 KB (1024-aligned)
    uint8_t *b_st = a_st + RA * kAStageBytes;            // RB x Mp*128 B (1024-aligned)
    uint8_t *w_st = b_st + RB * b_stage_bytes;           // RW x 12 KB (1024-aligned)
    uint64_t *w_full = reinterpret_cast<uint64_t *>(w_st + RW * kWStageBytes);
    uint64_t *w_empty = w_full + RW;
    uint64_t *a_full = w_empty + RW;
    uint64_t *a_empty = a_full + RA;
    uint64_t *b_full = a_empty + RA;
    uint64_t *b_empty = b_full + RB;
    uint64_t *done = b_empty + RB;  // [2]: per accumulator buffer, one phase per piece using it
    uint64_t *fin = done + 2;        // the MMA warp's own last wait: every MMA it issued has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *arr_tt = abort_flag + 1;    // [2] row tiles of this range's partial first / last piece
    volatile int *arr_last = arr_tt + 2;      // [2] this CTA delivered the row tile's last piece

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Ranges of units u = row_tile*G + group; a piece is the part of a range
    // inside one row tile.
    const int G = (int)t.G;
    const int V = (int)g.ranges;
    const int64_t T = t.Np / 16;  // stripes
    // Without PERSIST the grid holds one CTA per range (see k_gemm_tc).
    const int stride = PERSIST ? (int)gridDim.x : V;
    // piece jj of range v: row tile tt0 + jj, groups [ga, gb) of it
    struct Range {
        int u0, u1, tt0, ga0, npieces;
    };
    auto range_at = [&](int v) -> Range {
        Range rg;
        rg.u0 = range_begin(v, g);
        rg.u1 = range_begin(v + 1, g);
        rg.tt0 = rg.u0 / G;
        rg.ga0 = rg.u0 - rg.tt0 * G;
        rg.npieces = rg.u1 > rg.u0 ? (rg.u1 - 1) / G - rg.tt0 + 1 : 0;
        return rg;
    };
    auto piece = [&](const Range &rg, int jj, int &tt, int &ga, int &gb) {
        tt = rg.tt0 + jj;
        ga = jj == 0 ? rg.ga0 : 0;
        const int e = rg.u1 - tt * G;
        gb = e < G ? e : G;
    };
    const uint32_t acc_cols = tp.tmem_cols / 2;

    // the descriptors of the first copies load while the barriers are set up
    if (lane == 0) {
        if (warp == kWProdWarp) {
            prefetch_tmap(&hmap);
            if (!g.nested8) prefetch_tmap(&lmap);
        } else if (warp == kBProdWarp) {
            prefetch_tmap(&tmap);
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < RW; ++i) {
            mbar_init(&w_full[i], 1);    // the producer's expect_tx
            mbar_init(&w_empty[i], 8);   // one arrival per stripe's decoder warp of the k-block
        }
        for (int i = 0; i < RA; ++i) {
            mbar_init(&a_full[i], 8);
            mbar_init(&a_empty[i], 1);   // tcgen05.commit
        }
        for (int i = 0; i < RB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        mbar_init(&done[0], 1);
        mbar_init(&done[1], 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        arr_tt[0] = arr_tt[1] = -1;
        arr_last[0] = arr_last[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWProdWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(tp.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch();

    if (warp < kDecWarps) {
        // ------------------------------------------------------------------
        // Decoders: per piece (row tile tt, groups [ga, gb)), warp w handles
        // stripe st = 8*tt + (w%8) on every k-block (8 decoder warps) or on
        // the k-blocks of parity w/8 (16 warps: tiles p = w/8 and w/8 + 2 of
        // every group): the tile's planes come from the weight ring, the BF16
        // tile goes to the A ring (K-major, 128-byte swizzle), escapes over
        // their slots.  Then the piece's epilogue.  Every decoder warp runs
        // every range, piece and named barrier, also after an abort.
        // ------------------------------------------------------------------
        const int gid = lane >> 2, q = lane & 3;
        const int sw = warp & 7, par = warp >> 3;
        const int rA = 16 * sw + gid, rB = rA + 8;
        const uint32_t c28 = g.c28, c16 = g.c16;
        const uint32_t vmask = g.nested8 ? 0xFFF0u : 0xFFFFu;  // escape bits kept
        const int n_esc = (int)t.n_esc;
        const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32*quarter..; half: 0 .. kDecWarps/4 - 1
        const int r = 32 * quarter + lane;               // epilogue row within the row tile
        const int chunks = Mp / 16;

        RingPos wp, ap;  // ring positions of this warp's next k-block
        wp.advance(par, RW);
        ap.advance(par, RA);
        int it = 0;   // ranges this CTA has done
        int jb = 0;   // pieces this CTA has done in earlier ranges
        for (int v = blockIdx.x; v < V; v += stride, ++it) {
            const Range rg = range_at(v);
            const int npieces = rg.npieces;
            bool ok = !*abort_flag;

            // Piece epilogue (after its MMAs completed).  A piece covering its
            // whole row tile is rounded and stored; any other piece goes to
            // FP32 slot v (the range's first piece) or v + V (its last), and
            // the row tile's arrival count goes up.  Every decoder warp runs
            // the same barriers whether or not the CTA has aborted.
            auto epilogue = [&](int jj) {
                int tt, ga, gb;
                piece(rg, jj, tt, ga, gb);
                const int J = jb + jj;  // the piece's number in this CTA: buffer J & 1
                if (ok && !__all_sync(kFull, mbar_wait(&done[J & 1], (uint32_t)((J >> 1) & 1), abort_flag, g.error)))
                    ok = false;
                tc_fence_after();
                const bool whole = ga == 0 && gb == G;
                const int64_t slot = jj == 0 ? v : (int64_t)v + V;
                const int64_t n = (int64_t)tt * 128 + r;
                if (ok) {
                    const uint32_t acc = tmem + (uint32_t)(J & 1) * acc_cols + ((uint32_t)(32 * quarter) << 16);
                    for (int c = half; c < chunks; c += kDecWarps / 4) {
                        float x[16];
                        tmem_ld16(acc + (uint32_t)(16 * c), x);
                        if (SILU && whole) {  // hidden unit 8*(n/16) + n%16 on the gate lanes
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const float y = silu_pair(x[k]);
                                const int m = 16 * c + k;
                                if (!(lane & 8) && n < t.N && m < g.M)
                                    g.Y[(int64_t)m * g.ldy + (n >> 4) * 8 + (n & 7)] = f32_to_bf16_rn(y);
                            }
                        } else if (whole) {
                            if (n < t.N) {
#pragma unroll
                                for (int k = 0; k < 16; ++k) {
                                    const int m = 16 * c + k;
                                    if (m < g.M) g.Y[(int64_t)m * g.ldy + n] = f32_to_bf16_rn(x[k]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) g.partials[(slot * Mp + 16 * c + k) * 128 + r] = x[k];
                        }
                    }
                    if (!whole) __threadfence();
                }
                // every TMEM read of this buffer is done before any decoder warp
                // hands the MMA warp a tile of the piece that reuses it
                tc_fence_before();
                asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
                if (!whole && threadIdx.x == 0 && !*abort_flag) {
                    const int k = jj == 0 ? 0 : 1;
                    const int va = range_of(tt * G, g), vb = range_of(tt * G + G - 1, g);
                    arr_tt[k] = tt;
                    arr_last[k] = atomicAdd(&g.counters[tt], 1) == vb - va;
                }
            };

            // Per-piece state read from memory: row bases and the group offsets
            // (lane l holds the offset of group gw0 + l: one coalesced load per 31
            // groups, no dependent load inside the loop).  The next piece's is
            // fetched during the current piece's last group.
            struct PieceMeta {
                uint32_t base2A, base2B;
                int ptrw;
            };
            auto load_window = [&](const int32_t *gptr, bool live, int first, int gb) -> int {
                const int gi = first + lane;
                int x = 0;
                if (live && gi <= gb) {
                    x = __ldg(gptr + gi);
                    x = x < 0 ? 0 : (x > n_esc ? n_esc : x);
                }
                return x;
            };
            auto fetch_meta = [&](int jj) -> PieceMeta {
                int tt, ga, gb;
                piece(rg, jj, tt, ga, gb);
                const int64_t st = (int64_t)tt * 8 + sw;
                const bool live = st < T;
                PieceMeta pm;
                pm.base2A = pm.base2B = 0;
                if (live) {
                    const int64_t nA = st * 16 + gid, nB = nA + 8;
                    pm.base2A = (nA < t.N ? (uint32_t)__ldg(t.base + nA) : 0u) * 0x00800080u;
                    pm.base2B = (nB < t.N ? (uint32_t)__ldg(t.base + nB) : 0u) * 0x00800080u;
                }
                pm.ptrw = load_window(t.esc_ptr + (live ? st : 0) * t.G, live, ga, gb);
                return pm;
            };

            PieceMeta meta = fetch_meta(0);
            for (int j = 0; j < npieces; ++j) {
                int tt, ga, gb;
                piece(rg, j, tt, ga, gb);
                const int nkb = 4 * (gb - ga);
                const int64_t st = (int64_t)tt * 8 + sw;
                const bool live = st < T;  // warp-uniform
                const uint32_t base2A = meta.base2A, base2B = meta.base2B;
                const int32_t *gptr = t.esc_ptr + (live ? st : 0) * t.G;
                int gw0 = ga, ptrw = meta.ptrw;
                auto bounds = [&](int gg, int &p0, int &p1) {
                    if (gg + 1 - gw0 >= 32) {  // slide the window (more than 30 groups per piece)
                        gw0 = gg;
                        ptrw = load_window(gptr, live, gw0, gb);
                    }
                    p0 = __shfl_sync(kFull, ptrw, gg - gw0);
                    p1 = __shfl_sync(kFull, ptrw, gg + 1 - gw0);
                    if (p1 < p0) p1 = p0;
                };
                EscBatch cur, nxt;
                cur.cnt = nxt.cnt = 0;
                cur.ent = nxt.ent = 0;
                cur.p0 = nxt.p0 = 0;
                if (live) {
                    int p0, p1;
                    bounds(ga, p0, p1);
                    cur = load_group_escapes(t, p0, p1, lane);
                    if (ga + 1 < gb) {
                        bounds(ga + 1, p0, p1);
                        nxt = load_group_escapes(t, p0, p1, lane);
                    }
                }
                uint32_t emask = live ? escape_tiles(cur, lane) : 0u;
                // Y and the workspace may belong to the previous kernel (the
                // first piece's metadata above reads only the W12 tensor)
                if (it == 0 && j == 0) grid_dep_wait();
                if (j >= 2) epilogue(j - 2);  // frees the accumulator buffer this piece uses
                const int last_g = gb - ga - 1;
                // Each piece holds a multiple of 4 k-blocks, so this warp's k-blocks of
                // the piece start at parity `par` and its ring positions carry over.
                for (int kb = par; kb < nkb && ok; kb += kPar, wp.advance(kPar, RW), ap.advance(kPar, RA)) {
                    const int p = kb & 3;  // tile of the group
                    if (kb >= 4 && p == par && live) {  // first tile of a new group for this warp
                        const int gg = ga + (kb >> 2);
                        cur = nxt;
                        emask = escape_tiles(cur, lane);
                        if (gg + 1 < gb) {
                            int p0, p1;
                            bounds(gg + 1, p0, p1);
                            nxt = load_group_escapes(t, p0, p1, lane);
                        }
                    }
                    if ((kb >> 2) == last_g && p == par && j + 1 < npieces) meta = fetch_meta(j + 1);
                    const int ws = wp.stage, as = ap.stage;
                    const uint32_t wph = wp.phase, aph = ap.phase;
                    // the whole warp leaves together, so no lane is left behind at a
                    // warp-wide instruction
                    if (!__all_sync(kFull, mbar_wait(&w_full[ws], wph, abort_flag, g.error))) {
                        ok = false;
                        break;
                    }
                    uint32_t dA[8], dB[8];
                    if (live) {
                        const uint8_t *W = w_st + ws * kWStageBytes;
                        const uint4 h0 = lds128(W + sw * 1024 + lane * 16),
                                    h1 = lds128(W + sw * 1024 + 512 + lane * 16);
                        // the nested 8-bit view reads no lo plane: records with zero low nibbles
                        const uint4 l =
                            g.nested8 ? make_uint4(0u, 0u, 0u, 0u) : lds128(W + 8192 + sw * 512 + lane * 16);
                        decode16_fma(h0, l.x, l.y, base2A, c28, c16, dA);
                        decode16_fma(h1, l.z, l.w, base2B, c28, c16, dB);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_empty[ws]);  // the planes are in registers
                    if (!__all_sync(kFull, mbar_wait(&a_empty[as], aph ^ 1u, abort_flag, g.error))) {
                        ok = false;
                        break;
                    }
                    if (live) {
                        uint8_t *A = a_st + as * kAStageBytes;
                        *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q)) = make_uint4(dA[0], dA[1], dA[2], dA[3]);
                        *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q + 1)) = make_uint4(dA[4], dA[5], dA[6], dA[7]);
                        *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q)) = make_uint4(dB[0], dB[1], dB[2], dB[3]);
                        *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q + 1)) = make_uint4(dB[4], dB[5], dB[6], dB[7]);
                        if ((emask >> p) & 1u) {  // escapes of this tile overwrite their slots
                            __syncwarp();
                            auto put = [&](uint32_t e) {
                                const int key = (int)(e >> 16);
                                const int rr = 16 * sw + ((key >> 6) & 15), jj = key & 63;
                                *reinterpret_cast<uint16_t *>(A + swz(rr, jj >> 3) + (jj & 7) * 2) =
                                    (uint16_t)(e & vmask);
                            };
                            if (cur.cnt <= 32) {
                                if (lane < cur.cnt && (int)(cur.ent >> 26) == p) put(cur.ent);
                            } else {
                                for (int b0 = 0; b0 < cur.cnt; b0 += 32) {
                                    const uint32_t e = (b0 + lane < cur.cnt) ? __ldg(t.esc + cur.p0 + b0 + lane) : 0u;
                                    if (b0 + lane < cur.cnt && (int)(e >> 26) == p) put(e);
                                }
                            }
                        }
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[as]);
                }
            }
            if (npieces >= 2) epilogue(npieces - 2);
            if (npieces >= 1) epilogue(npieces - 1);

            // thread 0 records the arrivals after each epilogue's barrier:
            // one more barrier makes the last ones visible to every warp
            asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
            // Row tiles whose last piece this CTA delivered: sum the pieces in
            // range order and store.  (Only range va can start before the row
            // tile; its piece there is its last one.)
            for (int k = 0; k < 2; ++k) {
                const int tt = arr_tt[k];
                if (tt < 0 || !arr_last[k] || *abort_flag) continue;
                __threadfence();
                const int va = range_of(tt * G, g), vb = range_of(tt * G + G - 1, g);
                const int64_t s0 = range_begin(va, g) < tt * G ? (int64_t)va + V : va;
                const int64_t n = (int64_t)tt * 128 + r;
                if (SILU) {
                    const bool valid = n < t.N;  // the same for a gate lane and its up lane (N % 16 == 0)
                    for (int c = half; c < chunks; c += kDecWarps / 4) {
                        float acc[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            acc[jj] = valid ? __ldcg(g.partials + (s0 * Mp + 16 * c + jj) * 128 + r) : 0.f;
                        for (int x = va + 1; x <= vb; ++x) {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                acc[jj] += valid ? __ldcg(g.partials + ((int64_t)x * Mp + 16 * c + jj) * 128 + r) : 0.f;
                        }
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const float y = silu_pair(acc[jj]);
                            if (!(lane & 8) && valid && 16 * c + jj < g.M)
                                g.Y[(int64_t)(16 * c + jj) * g.ldy + (n >> 4) * 8 + (n & 7)] = f32_to_bf16_rn(y);
                        }
                    }
                } else if (n < t.N) {
                    for (int c = half; c < chunks; c += kDecWarps / 4) {
                        float acc[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            acc[jj] = __ldcg(g.partials + (s0 * Mp + 16 * c + jj) * 128 + r);
                        for (int x = va + 1; x <= vb; ++x) {
                            float y[16];
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                y[jj] = __ldcg(g.partials + ((int64_t)x * Mp + 16 * c + jj) * 128 + r);
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) acc[jj] += y[jj];
                        }
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            if (16 * c + jj < g.M) g.Y[(int64_t)(16 * c + jj) * g.ldy + n] = f32_to_bf16_rn(acc[jj]);
                    }
                }
                if (threadIdx.x == 0) g.counters[tt] = 0;
            }
            // every decoder warp has read this range's arrivals before thread
            // 0 clears them for the next one
            asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
            if (threadIdx.x == 0) {
                arr_tt[0] = arr_tt[1] = -1;
                arr_last[0] = arr_last[1] = 0;
            }
            jb += npieces;
        }
    } else if (warp == kWProdWarp) {
        // ------------------------------------------------------------------
        // Weight planes: one k-block (8 tiles of 1.5 KB) per stage, with
        // tiled copies, up to RW k-blocks ahead of the decoders, unit after
        // unit of each range.  Reads only the W12 tensor, so it starts before
        // the previous kernel ends.
        // ------------------------------------------------------------------
        // The whole warp runs the loop (warp-uniform values stay in uniform
        // registers); one elected lane issues.
        int issued = 0;
        bool ok = true;
        RingPos wp;
        for (int v = blockIdx.x; v < V && ok; v += stride) {
            const Range rg = range_at(v);
            int tt = rg.tt0, grp = rg.ga0;
            for (int u = rg.u0; u < rg.u1 && ok; ++u) {
                for (int p = 0; p < 4; ++p, wp.advance(1, RW)) {
                    const int ws = wp.stage;
                    if (!__all_sync(kFull, mbar_wait(&w_empty[ws], wp.phase ^ 1u, abort_flag, g.error))) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        // the full box is counted, out-of-range stripes included (zero-filled)
                        mbar_expect_tx(&w_full[ws], g.nested8 ? 8192u : kWStageBytes);
                        uint8_t *dst = w_st + ws * kWStageBytes;
                        tma_load_4d(dst, &hmap, 4 * grp + p, tt * 8, &w_full[ws]);
                        if (!g.nested8) tma_load_4d(dst + 8192, &lmap, 4 * grp + p, tt * 8, &w_full[ws]);
                    }
                    __syncwarp();
                    ++issued;
                }
                if (++grp == G) {
                    grp = 0;
                    ++tt;
                }
            }
        }
        // the copies issued last must have landed before the CTA exits
        for (int i = issued > RW ? issued - RW : 0; i < issued; ++i)
            mbar_drain(&w_full[i % RW], (uint32_t)((i / RW) & 1), g.error);
    } else if (warp == kBProdWarp) {
        // ------------------------------------------------------------------
        // Activations: one TMA tile [Mp x 64] per k-block.
        // ------------------------------------------------------------------
        grid_dep_wait();  // A may be written by the previous kernel
        int issued = 0;
        bool ok = true;
        RingPos bp;
        for (int v = blockIdx.x; v < V && ok; v += stride) {
            const Range rg = range_at(v);
            int grp = rg.ga0;
            for (int u = rg.u0; u < rg.u1 && ok; ++u) {
                for (int p = 0; p < 4; ++p, bp.advance(1, RB)) {
                    const int stage = bp.stage;
                    if (!__all_sync(kFull, mbar_wait(&b_empty[stage], bp.phase ^ 1u, abort_flag, g.error))) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        mbar_expect_tx(&b_full[stage], b_stage_bytes);
                        tma_load_2d(b_st + stage * b_stage_bytes, &tmap, (4 * grp + p) * 64, 0, &b_full[stage]);
                    }
                    __syncwarp();
                    ++issued;
                }
                if (++grp == G) grp = 0;
            }
        }
        // the copies issued last must have landed before the CTA exits
        for (int i = issued > RB ? issued - RB : 0; i < issued; ++i)
            mbar_drain(&b_full[i % RB], (uint32_t)((i / RB) & 1), g.error);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------
        // MMA issue.  The accumulator restarts at each piece's first k-block;
        // after a piece's last k-block a commit completes `done`.
        // ------------------------------------------------------------------
        // The whole warp runs the loop; one elected lane issues the MMAs.
        if (g.test_stall)  // a wait that nothing completes: it runs out and aborts the CTA
            (void)__all_sync(kFull, mbar_wait(fin, 0, abort_flag, g.error));
        bool ok = true;
        RingPos ap, bp;
        int j = -1;  // the CTA's piece number
        for (int v = blockIdx.x; v < V; v += stride) {
            const Range rg = range_at(v);
            int grp = rg.ga0;
            for (int u = rg.u0; u < rg.u1 && ok; ++u) {
                const bool first = u == rg.u0 || grp == 0;
                const bool last = u + 1 == rg.u1 || grp + 1 == G;
                if (first) ++j;
                const uint32_t d = tmem + (uint32_t)(j & 1) * acc_cols;
                for (int p = 0; p < 4; ++p, ap.advance(1, RA), bp.advance(1, RB)) {
                    const int as = ap.stage, bs = bp.stage;
                    if (!__all_sync(kFull, mbar_wait(&a_full[as], ap.phase, abort_flag, g.error)) ||
                        !__all_sync(kFull, mbar_wait(&b_full[bs], bp.phase, abort_flag, g.error))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(a_st + as * kAStageBytes);
                    const uint32_t b0 = smem_addr(b_st + bs * b_stage_bytes);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma(d, smem_desc(a0 + 32 * kk), smem_desc(b0 + 32 * kk), tp.idesc,
                                 !(first && p == 0 && kk == 0));
                        umma_commit(&a_empty[as]);
                        umma_commit(&b_empty[bs]);
                        if (last && p == 3) umma_commit(&done[j & 1]);
                    }
                    __syncwarp();
                }
                if (++grp == G) grp = 0;
            }
        }
        // TMEM and the shared-memory operands stay allocated until every MMA
        // issued has completed (after an abort the decoders stop waiting)
        if (elect_one()) umma_commit(fin);
        __syncwarp();
        (void)__all_sync(kFull, mbar_drain(fin, 0, g.error));
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWProdWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tp.tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

size_t tc_smem_bytes(const TcParams &tp) {
    return 1024 + (size_t)tp.a_st * kAStageBytes + (size_t)tp.b_st * tp.Mp * 128 + (size_t)tp.w_st * kWStageBytes +
           (size_t)(2 * (tp.a_st + tp.w_st + tp.b_st) + 3) * 8 + 32;  // rings, barriers, flags
}

// Dynamic shared memory one CTA may use: all 227 KB with one CTA per SM;
// with two, half of the SM's 228 KB less the 1 KB each CTA reserves.
size_t tc_smem_budget(int ctas_per_sm) { return ctas_per_sm > 1 ? 227 * 1024 / 2 - 1024 : 227 * 1024; }

// Ring depths within the shared-memory budget: about 96 KB (24 KB with two
// CTAs per SM) of activation stages (2 to 6); 3 decoded-A stages (4 above
// Mp = 128, 2 with two CTAs per SM); and the rest for weight stages: the
// weight ring is what keeps HBM busy (a k-block's planes take a few
// microseconds to arrive under load).  An activation stage is freed only
// when its k-block's MMAs complete, so at Mp = 256 (32 KB a stage) two
// stages left the MMAs waiting on the refill from L2: three ran the four
// layers 10% faster, and a fourth decoded-A stage another 2.5% (five weight
// stages are still enough there).  Returns false if not even two weight
// stages fit.
bool tc_rings(TcParams &tp, int ctas_per_sm) {
    const size_t budget = tc_smem_budget(ctas_per_sm);
    const size_t bst = (size_t)tp.Mp * 128;
    tp.b_st = (int)((ctas_per_sm > 1 ? 24 : 96) * 1024 / bst);
    tp.b_st = tp.b_st < 2 ? 2 : (tp.b_st > 6 ? 6 : tp.b_st);
    tp.a_st = ctas_per_sm > 1 ? 2 : (tp.Mp > 128 ? 4 : 3);
    tp.w_st = 0;
    for (int w = kMaxStages; w >= 2; --w) {
        TcParams x = tp;
        x.w_st = w;
        if (tc_smem_bytes(x) <= budget) {
            tp.w_st = w;
            break;
        }
    }
    return tp.w_st >= 2;
}

// Split of the K groups over S chunks for a grid of at most `slots` CTAs:
// no more chunks than column groups (or 16), and S <= 0.1*K/Mpad, so that
// the FP32 partials (2*S*Mpad*N*4 bytes written and read back) stay within
// about half the weight bytes (1.5*N*K); at these sizes they live in L2.
// (A cap of 0.0375*K/Mpad left QKV and O at M = 128 with 40-56 CTAs; on
// GB300 0.1 ran M = 128 and 256 13-17% faster and M <= 64 the same.)
// Above Mpad = 128 the cap is 0.15*K/Mpad, as measured on GB300: O at
// M = 256 then runs 120 CTAs instead of 80, 12% faster (0.15 for every Mpad
// made QKV at M = 128 slower).
int64_t tc_split_for(int64_t T, int64_t G, int64_t Mp, int64_t K, int64_t slots) {
    int64_t S = slots / T;
    const int64_t traffic_cap = (int64_t)((Mp > 128 ? 0.15 : 0.1) * (double)K / (double)Mp);
    if (S > traffic_cap) S = traffic_cap;
    if (S > G) S = G;
    if (S > 16) S = 16;
    if (S < 1) S = 1;
    return S;
}

// the kernel of a launch: K-chunks or balanced ranges, plain or with the
// fused gate/up epilogue; K-chunks with the split-K sum in global memory or
// across a cluster
template <int D, bool Ranges, bool SILU, bool PERSIST, bool CLUSTER>
struct TcKernel {
    static constexpr auto fn = k_gemm_tc<D, SILU, PERSIST, CLUSTER>;
};
template <int D, bool SILU, bool PERSIST, bool CLUSTER>
struct TcKernel<D, true, SILU, PERSIST, CLUSTER> {
    static constexpr auto fn = k_gemm_tc_ranges<D, SILU, PERSIST>;
};

// Raises the kernel's shared-memory limit, once per kernel and device
// (several host threads may launch at once).
template <auto kern>
cudaError_t configure_smem(size_t budget, int dev) {
    static std::mutex configured_mutex;
    static int configured[64] = {0};
    std::lock_guard<std::mutex> lock(configured_mutex);
    if (dev < 0 || dev >= 64 || configured[dev] < (int)budget) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = (int)budget;
    }
    return cudaSuccess;
}

template <int D, bool Ranges, bool SILU, bool PERSIST, bool CLUSTER>
cudaError_t launch_one(const TensorView &t, const GemmArgs &g, const TcParams &tp, const CUtensorMap &map,
                           const CUtensorMap &hmap, const CUtensorMap &lmap, cudaStream_t s) {
    constexpr auto kern = TcKernel<D, Ranges, SILU, PERSIST, CLUSTER>::fn;
    const size_t smem = tc_smem_bytes(tp);
    const size_t budget = tc_smem_budget(Roles<D>::kCtasPerSm);
    if (smem > budget) return cudaErrorInvalidConfiguration;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = configure_smem<kern>(budget, dev);
    if (e != cudaSuccess) return e;
    // one CTA per range, or per (row tile, K-chunk) item; a capped grid
    // walks the same items in the same cut (the result does not change)
    int64_t blocks = Ranges ? g.ranges : ((t.Np + 127) / 128) * (int64_t)g.split;
    if (blocks == 0) return cudaSuccess;
    if (PERSIST) blocks = g.max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(Roles<D>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (g.overlap) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (CLUSTER) {  // the split's S CTAs of a row tile (consecutive items) form one cluster
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)g.split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, t, g, tp, map, hmap, lmap);
}

// Whether the K-chunk build can sum its split across clusters: 2..8 chunks
// (a portable cluster), the FP32 partial [Mpad][128] fits the dynamic shared
// memory, and every cluster of the grid can be resident at once (a grid that
// no longer fits in one wave would lose more than the sum saves).  The
// answer depends on (device, build, split, Mpad) and is cached.
template <int D, bool SILU>
bool cluster_split_ok(const TensorView &t, const GemmArgs &g, const TcParams &tp) {
    const int S = g.split;
    if (S < 2 || S > 8) return false;
    const size_t smem = tc_smem_bytes(tp);
    if (smem < 1024 + 512 * (size_t)tp.Mp) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const int64_t grid = ((t.Np + 127) / 128) * (int64_t)S;
    static std::mutex m;
    static int cached[64][9][17] = {};  // [device][split][Mpad / 16]: 0 unknown, else max resident clusters + 1
    const int mi = (int)(tp.Mp / 16);
    if (mi < 1 || mi > 16) return false;
    std::lock_guard<std::mutex> lock(m);
    int &c = cached[dev][S][mi];
    if (c == 0) {
        constexpr auto kern = TcKernel<D, false, SILU, false, true>::fn;
        if (configure_smem<kern>(tc_smem_budget(Roles<D>::kCtasPerSm), dev) != cudaSuccess) return false;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)S);
        cfg.blockDim = dim3(Roles<D>::kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        c = n + 1;
    }
    return (int64_t)(c - 1) * S >= grid;
}

// One CTA per item, or (max_ctas below the item count) a capped grid of
// CTAs that walk several items each; an uncapped K-chunk split sums across
// clusters where it can (bitwise the same result).
template <int D, bool Ranges, bool SILU>
cudaError_t launch_variant(const TensorView &t, const GemmArgs &g, const TcParams &tp, const CUtensorMap &map,
                           const CUtensorMap &hmap, const CUtensorMap &lmap, cudaStream_t s) {
    const int64_t items = Ranges ? g.ranges : ((t.Np + 127) / 128) * (int64_t)g.split;
    if (g.max_ctas > 0 && g.max_ctas < items)
        return launch_one<D, Ranges, SILU, true, false>(t, g, tp, map, hmap, lmap, s);
    if (!Ranges && cluster_split_ok<D, SILU>(t, g, tp))
        return launch_one<D, false, SILU, false, true>(t, g, tp, map, hmap, lmap, s);
    return launch_one<D, Ranges, SILU, false, false>(t, g, tp, map, hmap, lmap, s);
}

}  // namespace

int64_t gemm_tc_pad(int64_t M) { return (M + 15) / 16 * 16; }

// The work of one launch, from (M, N, K) and a forced split only (never the
// grid), so the summation order is fixed.  Two schemes:
//  * K-chunks (k_gemm_tc): S chunks of whole groups per 128-row tile, one CTA
//    each; with Mpad <= 128, a split over 2 x 152 slots (two CTAs per SM)
//    when its grid holds at least kTwoPerSmMinCtas CTAs, otherwise about one
//    CTA per SM on 152 SMs.  S <= column groups, <= 16, and <= 0.1*K/Mpad, so
//    that the FP32 partials (2*S*Mpad*N*4 bytes written and read) stay within
//    about half the weight bytes (1.5*N*K); at these sizes they live in L2.
//  * balanced ranges (k_gemm_tc_ranges): with Mpad > 128 and at least 16
//    units (row tile, group) per SM, 152 contiguous ranges of units, one CTA
//    per SM.  There the K-chunk grid runs in more than one wave or leaves SMs
//    idle (gate/up, 272 row tiles; down, 120 CTAs), and the range kernel was
//    20% faster on GB300; with fewer units per CTA its per-piece costs made
//    it slower.
// Returns the bytes of FP32 partials the launch needs (0: none).
int64_t gemm_tc_plan(int64_t M, int64_t N, int64_t K, int split_k, bool counters_ok, GemmArgs &g) {
    const int64_t T = (N + 127) / 128, G = groups_of(K), Mp = gemm_tc_pad(M), Np = (N + 15) / 16 * 16;
    const int64_t U = T * G;
    g.tc_ranges = false;
    g.ranges = 0;
    if (split_k == 0 && counters_ok && Mp > 128 && U >= 16 * W12_PLAN_SMS) {
        const int64_t V = W12_PLAN_SMS;
        g.seglen = (int)U, g.per = (int)V;
        g.q = (int)(U / V), g.rem = (int)(U % V);
        g.ranges = V;
        g.split = 1;
        g.tc_cps = 1;
        g.tc_ranges = true;
        for (int64_t v = 1; v < V; ++v) {  // any range boundary inside a row tile needs partials
            const int64_t b = v * g.q + (v < g.rem ? v : g.rem);
            if (b % G != 0) return 2 * V * Mp * 128 * 4;
        }
        return 0;
    }
    int64_t S = 1;
    int cps = 1;
    if (split_k > 0) {
        S = split_k;
        cps = (Mp <= 128 && T * S >= kTwoPerSmMinCtas) ? 2 : 1;
    } else if (T > 0 && G > 0) {
        S = tc_split_for(T, G, Mp, K, W12_PLAN_SMS);
        if (Mp <= 128) {
            const int64_t S2 = tc_split_for(T, G, Mp, K, 2 * W12_PLAN_SMS);
            if (T * S2 >= kTwoPerSmMinCtas) {
                S = S2;
                cps = 2;
            }
        }
    }
    if (G == 0) S = 1;
    if (S > G && G > 0) S = G;
    if (!counters_ok) S = 1;
    if (S == 1) cps = (Mp <= 128 && T >= kTwoPerSmMinCtas) ? 2 : 1;
    g.split = (int)S;
    g.tc_cps = cps;
    return S > 1 ? S * Np * Mp * 4 : 0;
}

cudaError_t launch_gemm_tc(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TcParams tp;
    tp.Mp = (int)gemm_tc_pad(g.M);
    const int cps = g.tc_cps;
    if (!tc_rings(tp, cps)) return cudaErrorInvalidConfiguration;
    // a power of two >= max(32, Mp) columns per accumulator; the range kernel keeps two
    tp.tmem_cols = 32;
    while (tp.tmem_cols < tp.Mp) tp.tmem_cols <<= 1;
    if (g.tc_ranges) tp.tmem_cols *= 2;
    tp.idesc = (1u << 4)                         // D: FP32
               | (1u << 7) | (1u << 10)          // A, B: BF16
               | ((uint32_t)(tp.Mp >> 3) << 17)  // N
               | ((uint32_t)(128 >> 4) << 24);   // M = 128
    CUtensorMap map;
    const int64_t K = t.K > 0 ? t.K : 1;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)g.M};
    const cuuint64_t strides[1] = {(cuuint64_t)g.lda * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)tp.Mp};
    const cuuint32_t estr[2] = {1, 1};
    // with K = 0 the kernel issues no copy and the map is never read
    if (t.K > 0) {
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(g.A), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    } else {
        memset(&map, 0, sizeof map);
    }
    // The planes as 4-D u8 tensors [stripes][k-blocks][rows of 256 B][256 B].
    CUtensorMap hmap, lmap;
    {
        const cuuint64_t T = (cuuint64_t)(t.Np / 16), KT = (cuuint64_t)(t.KT > 0 ? t.KT : 1);
        const cuuint32_t e4[4] = {1, 1, 1, 1};
        const cuuint64_t hd[4] = {256, 4, KT, T}, hs[3] = {256, 1024, KT * 1024};
        const cuuint32_t hb[4] = {256, 4, 1, 8};
        const cuuint64_t ld[4] = {256, 2, KT, T}, ls[3] = {256, 512, KT * 512};
        const cuuint32_t lb[4] = {256, 2, 1, 8};
        if (t.K > 0) {
            CUresult r = enc(&hmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(t.hi), hd, hs, hb, e4,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
            r = enc(&lmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(t.lo), ld, ls, lb, e4,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        } else {
            memset(&hmap, 0, sizeof hmap);
            memset(&lmap, 0, sizeof lmap);
        }
    }
    if (g.silu) {
        if (g.tc_ranges) return launch_variant<16, true, true>(t, g, tp, map, hmap, lmap, s);
        return cps > 1 ? launch_variant<8, false, true>(t, g, tp, map, hmap, lmap, s)
                       : launch_variant<16, false, true>(t, g, tp, map, hmap, lmap, s);
    }
    if (g.tc_ranges) return launch_variant<16, true, false>(t, g, tp, map, hmap, lmap, s);
    return cps > 1 ? launch_variant<8, false, false>(t, g, tp, map, hmap, lmap, s)
                   : launch_variant<16, false, false>(t, g, tp, map, hmap, lmap, s);
}

}  // namespace w12
