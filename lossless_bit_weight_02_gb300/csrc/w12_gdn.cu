// Gated delta rule along the root paths of a draft tree: the recurrent-layer
// part of tree verification on hybrid models (SpecPilot, arXiv 2611.02501:
// the news article's part (2), Gated DeltaNet layers; the English summary's
// section 4.2 bullet on hybrid targets: a node's state is recomputed from the
// root state along its root path, and a WY kernel turns that chain of
// rank-one updates into matrix products on tensor cores, differing from the
// path kernel only in rounding).
//
// Per head, with the state S a D x D FP32 matrix (row = value index, column
// = key index), every node t of a root path applies
//     S <- alpha_t S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
// and a node's output is o = S q after its own update (the published gated
// delta rule; the pages name the layer but do not write it out).
//
// Two kernels compute the same outputs:
//   * k_gdn_path (the path kernel): one CTA per (node, head) starts from S_0
//     and applies the updates of the node's root path one by one.  Thread
//     pair (r, 0/1) holds half of row r of S in registers.
//   * the WY pair: with gamma the product of alpha along a path and f_t the
//     rank-one coefficient vectors,
//         f_t = beta_t (v_t - gamma_t S_0 k_t - sum_{j<t} G_tj (k_t.k_j) f_j)
//         o_t = gamma_t S_0 q_t + sum_{j<=t} G_tj (q_t.k_j) f_j
//     (j over the path's nodes, G_tj = product of alpha over the nodes after
//     j down to t).  S_0 enters only through K S_0^T and Q S_0^T for every
//     node at once: k_gdn_proj computes them with mma.sync (BF16 operands,
//     S_0 split into a BF16 high and low part so that the product keeps
//     FP32-level accuracy).  k_gdn_wy_paths then gives every (node, head) a
//     warp that recomputes the f of its own root path (no stored state, no
//     exchange between warps): the path keys' Gram matrix from mma.sync, a
//     forward substitution of at most 16 steps, and the output sum.
// Every sum runs in a fixed order, so both kernels are deterministic.
// Invalid trees (a parent outside [-1, i), a parent in another request, a
// request id outside [0, R), a path longer than 16) give NaN outputs for the
// nodes concerned and set the workspace error word.
#include <cstdint>
#include <cuda_runtime.h>

#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

constexpr int kGdnMaxDepth = W12_GDN_MAX_DEPTH;  // nodes on a root path
constexpr int kGdnMaxNodes = W12_GDN_MAX_NODES;  // nodes in one call

struct GdnArgs {
    const float *S0;                 // [R][H][D][D]
    const uint16_t *q, *k, *v;       // [n][H][D] BF16 bits
    const float *alpha, *beta;       // [n][H]
    const int32_t *parent;           // [n]
    const int32_t *req;              // [n] or null (every node in request 0)
    int n, H, R;
    float *o;                        // [n][H][D]
    int32_t *err;                    // workspace error word
    float *G;                        // [2][n][H][D]: K S_0^T, Q S_0^T (WY only)
    int32_t *paths;                  // [n][17]: path length (0 = invalid), then the path, node side first (WY only)
};

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ int req_of(const GdnArgs &a, int i) { return a.req ? a.req[i] : 0; }

// Node i's root path, node side first: up[0] = i, up[1] = its parent, ...
// Returns the length, or 0 if the chain is not a valid path of at most
// kGdnMaxDepth nodes inside one request.
template <typename Idx>
__device__ int walk_up(const GdnArgs &a, int i, Idx *up) {
    const int r = req_of(a, i);
    if (r < 0 || r >= a.R) return 0;
    int cur = i, L = 0;
    while (cur >= 0) {
        if (L == kGdnMaxDepth) return 0;
        up[L++] = (Idx)cur;
        const int p = a.parent[cur];
        if (p < -1 || p >= cur) return 0;
        if (p >= 0 && req_of(a, p) != r) return 0;
        cur = p;
    }
    return L;
}

// Warp sum with a fixed butterfly: every lane gets the same bits.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(kFull, x, s);
    return x;
}

// ---------------------------------------------------------------------------
// Path kernel.  Thread 2r + hf owns row r, columns col(j) = 8(j/4) + 4hf + j%4
// (j < D/2), so that the two threads of a row read different banks.
// ---------------------------------------------------------------------------
template <int D>
__global__ __launch_bounds__(2 * D, 2) void k_gdn_path(GdnArgs a) {
    constexpr int C = D / 2;
    __shared__ int up[kGdnMaxDepth];
    __shared__ int L_s;
    __shared__ float kv[2][D];  // k_t and v_t of the current step (then q)
    const int i = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int r = tid >> 1, hf = tid & 1;
    if (tid == 0) L_s = walk_up(a, i, up);
    __syncthreads();
    const int L = L_s;
    float *out = a.o + ((int64_t)i * a.H + h) * D;
    if (L == 0) {
        if (hf == 0) out[r] = __int_as_float(0x7FC00000);
        if (tid == 0) atomicExch(a.err, 1);
        return;
    }
    float S[C];
    {
        const float4 *row = reinterpret_cast<const float4 *>(
            a.S0 + (((int64_t)req_of(a, i) * a.H + h) * D + r) * D);
#pragma unroll
        for (int m = 0; m < C / 4; ++m) {
            const float4 x = row[2 * m + hf];
            S[4 * m] = x.x;
            S[4 * m + 1] = x.y;
            S[4 * m + 2] = x.z;
            S[4 * m + 3] = x.w;
        }
    }
    auto dot_row = [&](const float *x) {  // row r of S times x, halves added in a fixed order
        float p = 0.f;
#pragma unroll
        for (int j = 0; j < C; ++j) p = fmaf(S[j], x[8 * (j >> 2) + 4 * hf + (j & 3)], p);
        const float other = __shfl_xor_sync(kFull, p, 1);
        return hf ? other + p : p + other;
    };
    for (int s = L - 1; s >= 0; --s) {  // root side first
        const int t = up[s];
        const int64_t tb = ((int64_t)t * a.H + h) * D;
        if (tid < D) kv[0][tid] = bf2f(a.k[tb + tid]);
        else kv[1][tid - D] = bf2f(a.v[tb + tid - D]);
        const float al = a.alpha[(int64_t)t * a.H + h], be = a.beta[(int64_t)t * a.H + h];
        __syncthreads();
        const float u = dot_row(kv[0]);             // (S k)_r
        const float fr = be * (kv[1][r] - al * u);  // beta (v - alpha S k)_r
#pragma unroll
        for (int j = 0; j < C; ++j) S[j] = fmaf(fr, kv[0][8 * (j >> 2) + 4 * hf + (j & 3)], al * S[j]);
        __syncthreads();  // kv is rewritten next
    }
    if (tid < D) kv[0][tid] = bf2f(a.q[((int64_t)i * a.H + h) * D + tid]);
    __syncthreads();
    const float y = dot_row(kv[0]);
    if (hf == 0) out[r] = y;
}

// ---------------------------------------------------------------------------
// WY, step 1: G[0] = K S_0^T and G[1] = Q S_0^T for every node and head.
// One CTA per (request, head) lists the request's nodes (the head-0 CTA also
// walks and checks their root paths for step 2), loads S_0 once, split into
// BF16 hi + lo parts in shared memory (row pitch D + 8: conflict-free
// fragment reads), and its warps take 16-node tiles of K or Q:
// acc += X hi^T, then acc += X lo^T, per 16-wide k step, for all D columns.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two FP32 values as BF16 pairs: the nearest BF16 (hi) and the BF16 nearest
// to what remains (lo); lower column in the low half.
__device__ __forceinline__ void split2(float2 x, uint32_t &hi, uint32_t &lo) {
    const uint16_t h0 = f32_to_bf16_rn(x.x), h1 = f32_to_bf16_rn(x.y);
    const uint16_t l0 = f32_to_bf16_rn(x.x - bf2f(h0)), l1 = f32_to_bf16_rn(x.y - bf2f(h1));
    hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
    lo = (uint32_t)l0 | ((uint32_t)l1 << 16);
}

constexpr int kProjWarps = 8;

template <int D>
__host__ __device__ constexpr int proj_smem_bytes() {
    return 2 * D * (D + 8) * 2 + 4 * kGdnMaxNodes + 16;
}

template <int D>
__global__ __launch_bounds__(32 * kProjWarps) void k_gdn_proj(GdnArgs a) {
    constexpr int KP = D + 8, RW = KP / 2;  // BF16 row pitch, in u32
    extern __shared__ __align__(16) uint8_t smem_proj[];
    uint16_t *hi = reinterpret_cast<uint16_t *>(smem_proj);  // [D][KP]: row c = S_0 row c (value index)
    uint16_t *lo = hi + D * KP;
    int *list = reinterpret_cast<int *>(lo + D * KP);         // nodes of this request
    int *cnt = list + kGdnMaxNodes;
    const int r = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q4 = lane & 3;
    if (tid == 0) *cnt = 0;
    __syncthreads();
    // the nodes of request r (their order does not matter: MMA rows are independent)
    for (int i = tid; i < a.n; i += 32 * kProjWarps)
        if (req_of(a, i) == r) list[atomicAdd(cnt, 1)] = i;
    __syncthreads();
    const int nr = *cnt, tiles = (nr + 15) / 16;
    if (nr == 0) return;  // CTA-uniform
    if (h == 0) {  // every node's root path, once per request, for the per-path kernel
        for (int x = tid; x < nr; x += 32 * kProjWarps) {
            const int i = list[x];
            int32_t *pw = a.paths + (int64_t)i * 17;
            pw[0] = walk_up(a, i, pw + 1);
        }
    }
    // S_0[r][h] into the two BF16 parts (coalesced 16-byte loads, all in flight)
    const float4 *S0 = reinterpret_cast<const float4 *>(a.S0 + ((int64_t)r * a.H + h) * D * D);
#pragma unroll
    for (int it = 0; it < D * D / 4 / (32 * kProjWarps); ++it) {
        const int x = tid + 32 * kProjWarps * it;
        const float4 v4 = S0[x];
        const int c = (4 * x) / D, kk = (4 * x) % D;
        uint32_t h0, l0, h1, l1;
        split2(make_float2(v4.x, v4.y), h0, l0);
        split2(make_float2(v4.z, v4.w), h1, l1);
        *reinterpret_cast<uint2 *>(hi + c * KP + kk) = make_uint2(h0, h1);
        *reinterpret_cast<uint2 *>(lo + c * KP + kk) = make_uint2(l0, l1);
    }
    __syncthreads();
    const uint32_t *H32 = reinterpret_cast<const uint32_t *>(hi), *L32 = reinterpret_cast<const uint32_t *>(lo);
    for (int item = warp; item < 2 * tiles; item += kProjWarps) {
        const int tile = item >> 1, which = item & 1;
        const uint16_t *X = which ? a.q : a.k;
        const int iA = 16 * tile + g, iB = iA + 8;
        const bool okA = iA < nr, okB = iB < nr;
        const int rA = okA ? list[iA] : 0, rB = okB ? list[iB] : 0;
        const uint32_t *xa = reinterpret_cast<const uint32_t *>(X + ((int64_t)rA * a.H + h) * D);
        const uint32_t *xb = reinterpret_cast<const uint32_t *>(X + ((int64_t)rB * a.H + h) * D);
        uint32_t af[D / 16][4];
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
            const int w0 = 8 * s + q4;
            af[s][0] = okA ? xa[w0] : 0u;
            af[s][1] = okB ? xb[w0] : 0u;
            af[s][2] = okA ? xa[w0 + 4] : 0u;
            af[s][3] = okB ? xb[w0 + 4] : 0u;
        }
        float *G = a.G + (int64_t)which * a.n * a.H * D;
#pragma unroll 1
        for (int nt0 = 0; nt0 < D / 8; nt0 += 4) {  // four 8-column tiles at a time
            float acc[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[u][e] = 0.f;
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const int w0 = 8 * s + q4;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = (nt0 + u) * 8 + g;
                    mma_bf16(acc[u], af[s][0], af[s][1], af[s][2], af[s][3], H32[c * RW + w0], H32[c * RW + w0 + 4]);
                    mma_bf16(acc[u], af[s][0], af[s][1], af[s][2], af[s][3], L32[c * RW + w0], L32[c * RW + w0 + 4]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = (nt0 + u) * 8 + 2 * q4;
                if (okA) *reinterpret_cast<float2 *>(G + ((int64_t)rA * a.H + h) * D + c) = make_float2(acc[u][0], acc[u][1]);
                if (okB) *reinterpret_cast<float2 *>(G + ((int64_t)rB * a.H + h) * D + c) = make_float2(acc[u][2], acc[u][3]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// WY, step 2: one warp per (node, head) recomputes the coefficient vectors f
// of its own root path (up to 16; walked and checked by step 1) from the
// step-1 products, with no state and no exchange between warps:
//   * the path's keys go to shared memory as a 16 x D BF16 matrix Kp (rows
//     past the path are zero); their Gram matrix Kp Kp^T comes from
//     mma.sync (2 n-tiles x D/16 k-steps) and q_i . k_j from warp sums, and
//     then the f vectors take the keys' place in shared memory;
//   * w_t = v_t - gamma_t (K S_0^T)_t for every path node, then, root side
//     first, f_t = beta_t (w_t - sum_{j<t} G_tj Gram_tj f_j), j descending
//     (G_tj = alpha_{j+1} ... alpha_t, a running product);
//   * o = gamma (Q S_0^T)_i + sum_j G_ij (q_i.k_j) f_j, j descending.
// Lane l holds columns l, l + 32, ... of every vector.
// ---------------------------------------------------------------------------
constexpr int kPathWarps = 4;  // warps (nodes) per CTA
static_assert(kGdnMaxDepth == 16, "a root path fills the 16 rows of one m16n8k16 tile");

template <int D>
__host__ __device__ constexpr int path_warp_bytes() {
    // the path keys (BF16, until their products are formed) and then the f
    // vectors (FP32) share the first region
    return (16 * (D + 8) * 2 > 16 * D * 4 ? 16 * (D + 8) * 2 : 16 * D * 4) + 16 * 17 * 4 + 5 * 16 * 4;
}

template <int D>
__global__ __launch_bounds__(32 * kPathWarps) void k_gdn_wy_paths(GdnArgs a) {
    constexpr int P = D / 32, KP = D + 8;
    extern __shared__ __align__(16) uint8_t smem_gdn[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;
    const int i = blockIdx.x * kPathWarps + warp, h = blockIdx.y;
    if (i >= a.n) return;  // warp-uniform; the kernel has no block barrier
    uint8_t *base = smem_gdn + warp * path_warp_bytes<D>();
    constexpr int kRegion = 16 * (D + 8) * 2 > 16 * D * 4 ? 16 * (D + 8) * 2 : 16 * D * 4;
    uint16_t *Kp = reinterpret_cast<uint16_t *>(base);  // [16][KP], then
    float *fs = reinterpret_cast<float *>(base);        // [16][D] over it
    float *gram = reinterpret_cast<float *>(base + kRegion);  // [16][17]
    float *al = gram + 16 * 17, *be = al + 16, *gm = be + 16, *qk = gm + 16;  // [16] each
    int *up = reinterpret_cast<int *>(qk + 16);                                 // [16]
    const int64_t ih = ((int64_t)i * a.H + h) * D;
    const float *G2 = a.G + (int64_t)a.n * a.H * D;
    float qi[P], g2[P];
#pragma unroll
    for (int m = 0; m < P; ++m) {
        qi[m] = bf2f(a.q[ih + lane + 32 * m]);
        g2[m] = G2[ih + lane + 32 * m];
    }
    // the root path, walked and checked once per request by the projection
    // kernel (a node with a bad request id is in no request's list)
    const int rq = req_of(a, i);
    int L = 0;
    if (rq >= 0 && rq < a.R) {
        const int32_t *pw = a.paths + (int64_t)i * 17;
        L = pw[0];
        if (lane < L) up[lane] = pw[1 + lane];
    }
    __syncwarp();
    float *out = a.o + ih;
    if (L == 0) {
#pragma unroll
        for (int m = 0; m < P; ++m) out[lane + 32 * m] = __int_as_float(0x7FC00000);
        if (lane == 0) atomicExch(a.err, 1);
        return;
    }
    // path node t (root side first) is up[L - 1 - t].  The path's alpha and
    // beta and the key rows are all requested here.
    if (lane < 16) {
        const int node = lane < L ? up[L - 1 - lane] : 0;
        al[lane] = lane < L ? a.alpha[(int64_t)node * a.H + h] : 0.f;
        be[lane] = lane < L ? a.beta[(int64_t)node * a.H + h] : 0.f;
    }
    constexpr int CH = D / 8;  // 16-byte chunks per key row
#pragma unroll
    for (int it = 0; it < 16 * CH / 32; ++it) {
        const int c = lane + 32 * it, t = c / CH, ch = c - t * CH;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (t < L) x = *reinterpret_cast<const uint4 *>(a.k + ((int64_t)up[L - 1 - t] * a.H + h) * D + 8 * ch);
        *reinterpret_cast<uint4 *>(Kp + t * KP + 8 * ch) = x;
    }
    __syncwarp();
    if (lane < 16) {  // gamma_t = alpha_0 ... alpha_t
        float gam = 1.f;
        for (int t = 0; t <= lane; ++t) gam *= al[t];
        gm[lane] = gam;
    }
    __syncwarp();
    // Gram = Kp Kp^T
    {
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        const uint32_t *K32 = reinterpret_cast<const uint32_t *>(Kp);
        constexpr int RW = KP / 2;  // u32 per row
#pragma unroll
        for (int kk = 0; kk < D; kk += 16) {
            const int w0 = (kk >> 1) + q4;
            const uint32_t a0 = K32[g * RW + w0], a1 = K32[(g + 8) * RW + w0];
            const uint32_t a2 = K32[g * RW + w0 + 4], a3 = K32[(g + 8) * RW + w0 + 4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int rn = nt * 8 + g;
                mma_bf16(acc[nt], a0, a1, a2, a3, K32[rn * RW + w0], K32[rn * RW + w0 + 4]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            gram[g * 17 + nt * 8 + 2 * q4] = acc[nt][0];
            gram[g * 17 + nt * 8 + 2 * q4 + 1] = acc[nt][1];
            gram[(g + 8) * 17 + nt * 8 + 2 * q4] = acc[nt][2];
            gram[(g + 8) * 17 + nt * 8 + 2 * q4 + 1] = acc[nt][3];
        }
    }
    // q_i . k_j for the path's keys
    for (int j = 0; j < L; ++j) {
        float pq = 0.f;
#pragma unroll
        for (int m = 0; m < P; ++m) pq = fmaf(qi[m], bf2f(Kp[j * KP + lane + 32 * m]), pq);
        pq = warp_sum(pq);
        if (lane == 0) qk[j] = pq;
    }
    __syncwarp();  // the keys are no longer read: fs takes their place
    // w_t = v_t - gamma_t (K S_0^T)_t into fs, four columns per chunk
#pragma unroll 8
    for (int it = 0; it < 16 * (D / 4) / 32; ++it) {
        const int x = lane + 32 * it, t = x / (D / 4), c = 4 * (x % (D / 4));
        if (t < L) {
            const int64_t th = ((int64_t)up[L - 1 - t] * a.H + h) * D + c;
            const float4 g1 = *reinterpret_cast<const float4 *>(a.G + th);
            const uint2 vv = *reinterpret_cast<const uint2 *>(a.v + th);
            const float gam = gm[t];
            *reinterpret_cast<float4 *>(fs + t * D + c) =
                make_float4(__uint_as_float(vv.x << 16) - gam * g1.x, __uint_as_float(vv.x & 0xFFFF0000u) - gam * g1.y,
                            __uint_as_float(vv.y << 16) - gam * g1.z, __uint_as_float(vv.y & 0xFFFF0000u) - gam * g1.w);
        }
    }
    __syncwarp();
    // f_t, root side first
    for (int t = 0; t < L; ++t) {
        float s[P];
#pragma unroll
        for (int m = 0; m < P; ++m) s[m] = 0.f;
        float r = 1.f;
        for (int j = t - 1; j >= 0; --j) {
            r *= al[j + 1];
            const float cf = r * gram[t * 17 + j];
#pragma unroll
            for (int m = 0; m < P; ++m) s[m] = fmaf(cf, fs[j * D + lane + 32 * m], s[m]);
        }
        const float bt = be[t];
#pragma unroll
        for (int m = 0; m < P; ++m) fs[t * D + lane + 32 * m] = bt * (fs[t * D + lane + 32 * m] - s[m]);
        __syncwarp();
    }
    // output of node i (path node L - 1)
    float o[P];
    const float gam = gm[L - 1];
#pragma unroll
    for (int m = 0; m < P; ++m) o[m] = 0.f;
    float r = 1.f;
    for (int j = L - 1; j >= 0; --j) {
        if (j < L - 1) r *= al[j + 1];
        const float cf = r * qk[j];
#pragma unroll
        for (int m = 0; m < P; ++m) o[m] = fmaf(cf, fs[j * D + lane + 32 * m], o[m]);
    }
#pragma unroll
    for (int m = 0; m < P; ++m) out[lane + 32 * m] = fmaf(gam, g2[m], o[m]);
}

template <int D>
cudaError_t launch_gdn_d(const GdnArgs &a, int mode, cudaStream_t s) {
    if (mode == 0) {
        k_gdn_path<D><<<dim3((unsigned)a.n, (unsigned)a.H), 2 * D, 0, s>>>(a);
        return cudaGetLastError();
    }
    constexpr int smem = kPathWarps * path_warp_bytes<D>(), psmem = proj_smem_bytes<D>();
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(k_gdn_wy_paths<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_gdn_proj<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    k_gdn_proj<D><<<dim3((unsigned)a.R, (unsigned)a.H), 32 * kProjWarps, psmem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_gdn_wy_paths<D><<<dim3((unsigned)((a.n + kPathWarps - 1) / kPathWarps), (unsigned)a.H), 32 * kPathWarps,
                         smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t gdn_workspace_bytes(int64_t n, int64_t H, int64_t D, int mode) {
    if (mode == 0) return 256;
    return 256 + (size_t)2 * (size_t)n * (size_t)H * (size_t)D * 4 + ((size_t)n * 17 * 4 + 15) / 16 * 16;
}

cudaError_t launch_gdn_tree(const float *S0, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *alpha, const float *beta, const int32_t *parent, const int32_t *req,
                            int n, int H, int R, int D, float *o, void *workspace, int mode, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, 4, s);
    if (e != cudaSuccess || n == 0) return e;
    GdnArgs a;
    a.S0 = S0;
    a.q = q;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.parent = parent;
    a.req = req;
    a.n = n;
    a.H = H;
    a.R = R;
    a.o = o;
    a.err = static_cast<int32_t *>(workspace);
    a.G = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + 256);
    a.paths = reinterpret_cast<int32_t *>(a.G + (int64_t)2 * n * H * D);
    if (D == 64) return launch_gdn_d<64>(a, mode, s);
    if (D == 128) return launch_gdn_d<128>(a, mode, s);
    return cudaErrorInvalidValue;
}

}  // namespace w12
