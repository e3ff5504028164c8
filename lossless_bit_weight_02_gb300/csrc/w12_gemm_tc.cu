// W12 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM) for
// 16 <= Mpad <= 256 tokens: Y = A * W^T with W decoded on the fly
// (SpecPilot, arXiv 2611.02501, section 4.1: the GEMM decodes the records in
// registers and splits its reduction in a fixed order).
//
// One CTA owns 128 weight rows (8 stripes of 16) and a chunk of whole
// 256-column groups; per 64-column k-block:
//   * 8 decoder warps (one stripe each) stream their tile (1.5 KB, the same
//     fragment-native loads as the small-M kernel, one 4-tile group in
//     flight), decode it in registers and store it as BF16 into the UMMA A
//     operand: 128 rows x 128 bytes, K-major, 128-byte swizzle.  Escapes of
//     the tile are written over their slots in shared memory.  Each thread
//     then fences the generic->async proxy and arrives on the stage's
//     "A full" barrier;
//   * one producer thread loads the activation tile [Mpad x 64] with TMA
//     (rows >= M and columns >= K come back as zeros) into the B operand;
//   * one MMA thread waits for both, issues four tcgen05.mma (M=128,
//     N=Mpad, K=16) accumulating in TMEM, and commits to the stage's "empty"
//     barrier.
// The epilogue warps read the accumulator with tcgen05.ld.  With a split of
// S > 1 the chunk partials go to the FP32 workspace and the last CTA of a row
// tile adds them in the order s = 0..S-1; S depends only on (M, N, K).
// Every mbarrier wait is bounded: on expiry the CTA records W12_ERR_TIMEOUT in
// the workspace error word, waits (bounded) for its own copies and MMAs, and
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

constexpr int kDecWarps = 16;     // two per 16-row stripe (even / odd tiles of each group)
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;      // the warp after the producer issues the MMAs
constexpr int kThreads = 32 * (kDecWarps + 2);
constexpr uint32_t kAStageBytes = 128 * 128;  // 128 rows x 64 BF16
constexpr long long kWaitPolls = 1LL << 20;    // each poll is a try_wait (which may itself block)

struct TcParams {
    int Mp;         // tokens padded to a multiple of 16 (UMMA N)
    int stages;     // pipeline depth
    int tmem_cols;  // power of two >= max(32, Mp)
    uint32_t idesc; // tcgen05 instruction descriptor
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
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the completion of phase `parity`.  Gives up (returns
// false) when another thread of the CTA has given up, or after kWaitPolls
// polls, in which case it raises the CTA's abort flag and the error word.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err) {
    for (long long i = 0; i < kWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort_flag) return false;
    }
    *abort_flag = 1;
    atomicExch(err, 1);
    return false;
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

// Byte offset of (row r, 16-byte chunk c) in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ __launch_bounds__(kThreads, 1) void k_gemm_tc(TensorView t, GemmArgs g, TcParams tp,
                                                         const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int R = tp.stages, Mp = tp.Mp;
    const uint32_t b_stage_bytes = (uint32_t)Mp * 128;
    uint8_t *a_st = base;
    uint8_t *b_st = base + R * kAStageBytes;
    uint64_t *full_a = reinterpret_cast<uint64_t *>(b_st + R * b_stage_bytes);
    uint64_t *full_b = full_a + R;
    uint64_t *empty = full_b + R;
    uint64_t *done = empty + R;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = g.split;
    const int64_t tt = blockIdx.x / S;  // 128-row tile
    const int s = (int)(blockIdx.x % S);
    const int64_t g_beg = (s * t.G) / S, g_end = ((s + 1) * t.G) / S;
    const int nkb = (int)(4 * (g_end - g_beg));

    if (threadIdx.x == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(&full_a[i], (kDecWarps / 2) * 32);  // the 8 warps of one tile parity
            mbar_init(&full_b[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kProducerWarp) {
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
        // Decoders: warp w handles stripe st = 8*tt + (w%8) and the tiles
        // p = w/8 and w/8 + 2 of every group.
        // ------------------------------------------------------------------
        const int gid = lane >> 2, q = lane & 3;
        const int sw = warp & 7, par = warp >> 3;
        const int64_t T = t.Np / 16;
        const int64_t st = tt * 8 + sw;
        const bool live = st < T;  // warp-uniform
        const int rA = 16 * sw + gid, rB = rA + 8;
        const uint32_t c28 = g.c28, c16 = g.c16;
        uint4 bh0[2], bh1[2], bl[2];
        const uint4 *hp = reinterpret_cast<const uint4 *>(t.hi) + (st * t.KT + 4 * g_beg + par) * 64 + lane;
        const uint4 *lp = reinterpret_cast<const uint4 *>(t.lo) + (st * t.KT + 4 * g_beg + par) * 32 + lane;
        uint32_t base2A = 0, base2B = 0;
        EscBatch cur, nxt;
        cur.cnt = nxt.cnt = 0;
        cur.ent = nxt.ent = 0;
        cur.p0 = nxt.p0 = 0;
        const int32_t *gptr = t.esc_ptr + (live ? st : 0) * t.G;
        const int n_esc = (int)t.n_esc;
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
        int ptrw = load_window(gw0);
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
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                bh0[i] = ld_stream(hp + i * 128);
                bh1[i] = ld_stream(hp + i * 128 + 32);
                bl[i] = ld_stream(lp + i * 64);
            }
            const int64_t nA = st * 16 + gid, nB = nA + 8;
            base2A = (nA < t.N ? (uint32_t)__ldg(t.base + nA) : 0u) * 0x00800080u;
            base2B = (nB < t.N ? (uint32_t)__ldg(t.base + nB) : 0u) * 0x00800080u;
            int p0, p1;
            bounds(g_beg, p0, p1);
            cur = load_group_escapes(t, p0, p1, lane);
            if (g_beg + 1 < g_end) {
                bounds(g_beg + 1, p0, p1);
                nxt = load_group_escapes(t, p0, p1, lane);
            }
        }
        uint32_t emask = (live && nkb > 0) ? escape_tiles(cur, lane) : 0u;
        grid_dep_wait();  // Y and the workspace may belong to the previous kernel
        bool ok = true;
        for (int64_t gg = g_beg; gg < g_end && ok; ++gg) {
            const bool more = gg + 1 < g_end;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int p = par + 2 * i;  // tile of the group
                const int kb = (int)(4 * (gg - g_beg)) + p;
                const int stage = kb % R;
                const uint32_t ph = (uint32_t)((kb / R) & 1);
                uint32_t dA[8], dB[8];
                if (live) {
                    decode16_fma(bh0[i], bl[i].x, bl[i].y, base2A, c28, c16, dA);
                    decode16_fma(bh1[i], bl[i].z, bl[i].w, base2B, c28, c16, dB);
                    if (more) {
                        bh0[i] = ld_stream(hp + 256 + i * 128);
                        bh1[i] = ld_stream(hp + 256 + i * 128 + 32);
                        bl[i] = ld_stream(lp + 128 + i * 64);
                    }
                }
                // the whole warp leaves together, so no lane is left behind at
                // a warp-wide instruction
                if (!__all_sync(kFull, mbar_wait(&empty[stage], ph ^ 1u, abort_flag, g.error))) {
                    ok = false;
                    break;
                }
                if (live) {
                    uint8_t *A = a_st + stage * kAStageBytes;
                    *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q)) = make_uint4(dA[0], dA[1], dA[2], dA[3]);
                    *reinterpret_cast<uint4 *>(A + swz(rA, 2 * q + 1)) = make_uint4(dA[4], dA[5], dA[6], dA[7]);
                    *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q)) = make_uint4(dB[0], dB[1], dB[2], dB[3]);
                    *reinterpret_cast<uint4 *>(A + swz(rB, 2 * q + 1)) = make_uint4(dB[4], dB[5], dB[6], dB[7]);
                    if ((emask >> p) & 1u) {  // escapes of this tile overwrite their slots
                        __syncwarp();
                        auto put = [&](uint32_t e) {
                            const int key = (int)(e >> 16);
                            const int r = 16 * sw + ((key >> 6) & 15), j = key & 63;
                            *reinterpret_cast<uint16_t *>(A + swz(r, j >> 3) + (j & 7) * 2) = (uint16_t)(e & 0xFFFFu);
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
                mbar_arrive(&full_a[stage]);
            }
            if (live) {
                hp += 256;
                lp += 128;
                cur = nxt;
                emask = more ? escape_tiles(cur, lane) : 0u;
                if (gg + 2 < g_end) {
                    int p0, p1;
                    bounds(gg + 2, p0, p1);
                    nxt = load_group_escapes(t, p0, p1, lane);
                }
            }
        }

        // ------------------------------------------------------------------
        // Epilogue: TMEM lanes 32*(warp%4).. ; the four warps w, w+4, w+8,
        // w+12 split the 16-column chunks.
        // ------------------------------------------------------------------
        const bool fin = __all_sync(kFull, mbar_wait(done, 0, abort_flag, g.error));
        tc_fence_after();
        const int quarter = warp & 3, half = warp >> 2;  // half: 0..3
        const int64_t n = tt * 128 + 32 * quarter + lane;
        const int chunks = Mp / 16;
        const bool have = __all_sync(kFull, fin && ok && !*abort_flag);
        if (have) {
            for (int c = half; c < chunks; c += 4) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(16 * c), v);
                if (nkb == 0) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
                if (S == 1) {
                    if (n < t.N) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * c + j;
                            if (m < g.M) g.Y[(int64_t)m * g.ldy + n] = f32_to_bf16_rn(v[j]);
                        }
                    }
                } else if (n < t.Np) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        g.partials[((int64_t)s * Mp + 16 * c + j) * t.Np + n] = v[j];
                }
            }
        }
        if (S > 1) {
            // fixed-order combination by the last CTA of this row tile
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
            if (threadIdx.x == 0) *last_flag = have ? (atomicAdd(&g.counters[tt], 1) == S - 1) : 0;
            asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
            if (*last_flag) {
                __threadfence();
                if (n < t.N) {
                    for (int c = half; c < chunks; c += 4) {
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * c + j;
                            if (m >= g.M) break;
                            float acc = __ldcg(g.partials + (int64_t)m * t.Np + n);
                            for (int ss = 1; ss < S; ++ss) acc += __ldcg(g.partials + ((int64_t)ss * Mp + m) * t.Np + n);
                            g.Y[(int64_t)m * g.ldy + n] = f32_to_bf16_rn(acc);
                        }
                    }
                }
                if (threadIdx.x == 0) g.counters[tt] = 0;
            }
        }
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------------
        // Activations: one TMA tile [Mp x 64] per k-block.
        // ------------------------------------------------------------------
        if (lane == 0) {
            grid_dep_wait();  // A may be written by the previous kernel
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int stage = kb % R;
                const uint32_t ph = (uint32_t)((kb / R) & 1);
                if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, g.error)) break;
                mbar_expect_tx(&full_b[stage], b_stage_bytes);
                tma_load_2d(b_st + stage * b_stage_bytes, &tmap, (int)((4 * g_beg + kb) * 64), 0, &full_b[stage]);
                ++issued;
            }
            // the copies issued last must have landed before the CTA exits
            for (int i = issued > R ? issued - R : 0; i < issued; ++i)
                mbar_wait(&full_b[i % R], (uint32_t)((i / R) & 1), abort_flag, g.error);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------
        // MMA issue (one thread).
        // ------------------------------------------------------------------
        if (lane == 0) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int stage = kb % R;
                const uint32_t ph = (uint32_t)((kb / R) & 1);
                if (!mbar_wait(&full_a[stage], ph, abort_flag, g.error)) break;
                if (!mbar_wait(&full_b[stage], ph, abort_flag, g.error)) break;
                tc_fence_after();
                const uint32_t a0 = smem_addr(a_st + stage * kAStageBytes);
                const uint32_t b0 = smem_addr(b_st + stage * b_stage_bytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma(tmem, smem_desc(a0 + 32 * kk), smem_desc(b0 + 32 * kk), tp.idesc, (kb | kk) != 0);
                umma_commit(&empty[stage]);
            }
            umma_commit(done);  // arrives once every MMA issued above has completed
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kProducerWarp) {
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

int tc_stages(int Mp) {  // one CTA per SM: up to ~200 KB of stages
    const int stage = (int)kAStageBytes + Mp * 128;
    int r = (200 * 1024) / stage;
    return r < 2 ? 2 : (r > 6 ? 6 : r);
}

size_t tc_smem_bytes(int Mp, int R) {
    return 1024 + (size_t)R * (kAStageBytes + (size_t)Mp * 128) + (size_t)(3 * R + 1) * 8 + 16;
}

}  // namespace

int64_t gemm_tc_pad(int64_t M) { return (M + 15) / 16 * 16; }

// Split from (M, N, K) only: about one CTA per SM on 152 SMs, no more chunks
// than column groups, and few enough that the FP32 partial traffic
// (2*S*Mpad*N*4 bytes) stays small next to the weights (1.5*N*K bytes).
int gemm_tc_split(int64_t M, int64_t N, int64_t K) {
    const int64_t T = (N + 127) / 128, G = groups_of(K), Mp = gemm_tc_pad(M);
    if (T == 0 || G == 0) return 1;
    int64_t S = 152 / T;
    const int64_t traffic_cap = (int64_t)(0.0375 * (double)K / (double)Mp);
    if (S > traffic_cap) S = traffic_cap;
    if (S > G) S = G;
    if (S > 16) S = 16;
    if (S < 1) S = 1;
    return (int)S;
}

cudaError_t launch_gemm_tc(const TensorView &t, const GemmArgs &g, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TcParams tp;
    tp.Mp = (int)gemm_tc_pad(g.M);
    tp.stages = tc_stages(tp.Mp);
    tp.tmem_cols = 32;
    while (tp.tmem_cols < tp.Mp) tp.tmem_cols <<= 1;
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
    const size_t smem = tc_smem_bytes(tp.Mp, tp.stages);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int configured[64] = {0};
    if (dev >= 0 && dev < 64 && configured[dev] < (int)smem) {
        e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = 227 * 1024;
    }
    const int64_t blocks = ((t.Np + 127) / 128) * (int64_t)g.split;
    if (blocks == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc, t, g, tp, map);
}

}  // namespace w12
