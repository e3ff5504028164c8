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
//     FP32-level accuracy).  k_gdn_wy_tree then walks the tree level by level
//     (one CTA per head, one warp per node), each node a few dot products and
//     vector sums of length D.
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

constexpr int kGdnMaxDepth = 16;
constexpr int kGdnMaxNodes = 1024;
constexpr int kTreeThreads = 512;

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
    float *f;                        // [n][H][D] (WY only)
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
// A CTA takes 16 nodes of one head and one of K / Q; warp w the output
// columns 32w .. 32w+31 (four m16n8 tiles).  S_0 = hi + lo, both BF16:
// acc += X hi^T, then acc += X lo^T, per 16-wide k step.  Rows of the tile
// that belong to different requests are done one request after another.
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

template <int D>
__global__ __launch_bounds__(D) void k_gdn_proj(GdnArgs a) {
    const int tile = blockIdx.x >> 1, which = blockIdx.x & 1, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;
    const uint16_t *X = which ? a.q : a.k;
    const int rA = tile * 16 + g, rB = rA + 8;
    const bool okA = rA < a.n, okB = rB < a.n;
    const int reqA = okA ? req_of(a, rA) : -1, reqB = okB ? req_of(a, rB) : -1;
    // requests still to do for this lane's two rows (an invalid id is never done)
    bool todoA = okA && reqA >= 0 && reqA < a.R, todoB = okB && reqB >= 0 && reqB < a.R;
    const uint32_t *xa = reinterpret_cast<const uint32_t *>(X + ((int64_t)(okA ? rA : 0) * a.H + h) * D);
    const uint32_t *xb = reinterpret_cast<const uint32_t *>(X + ((int64_t)(okB ? rB : 0) * a.H + h) * D);
    float *G = a.G + (int64_t)which * a.n * a.H * D;
    while (__any_sync(kFull, todoA || todoB)) {
        // the smallest request id still to do in the tile
        const unsigned mine = todoA ? (unsigned)reqA : (todoB ? (unsigned)reqB : 0xFFFFFFFFu);
        const unsigned mineB = todoB ? (unsigned)reqB : 0xFFFFFFFFu;
        const int rq = (int)__reduce_min_sync(kFull, mine < mineB ? mine : mineB);
        const float *S0 = a.S0 + ((int64_t)rq * a.H + h) * D * D;
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        for (int kk = 0; kk < D; kk += 16) {
            const int w0 = (kk >> 1) + q4;  // u32 index of columns kk + 2q4, +1
            const uint32_t a0 = okA ? xa[w0] : 0u, a1 = okB ? xb[w0] : 0u;
            const uint32_t a2 = okA ? xa[w0 + 4] : 0u, a3 = okB ? xb[w0 + 4] : 0u;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int c = warp * 32 + nt * 8 + g;  // output column = row c of S_0
                const float *srow = S0 + (int64_t)c * D + kk + 2 * q4;
                uint32_t h0, l0, h1, l1;
                split2(*reinterpret_cast<const float2 *>(srow), h0, l0);
                split2(*reinterpret_cast<const float2 *>(srow + 8), h1, l1);
                mma_bf16(acc[nt], a0, a1, a2, a3, h0, h1);
                mma_bf16(acc[nt], a0, a1, a2, a3, l0, l1);
            }
        }
        const bool wA = todoA && reqA == rq, wB = todoB && reqB == rq;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int c = warp * 32 + nt * 8 + 2 * q4;
            if (wA) *reinterpret_cast<float2 *>(G + ((int64_t)rA * a.H + h) * D + c) = make_float2(acc[nt][0], acc[nt][1]);
            if (wB) *reinterpret_cast<float2 *>(G + ((int64_t)rB * a.H + h) * D + c) = make_float2(acc[nt][2], acc[nt][3]);
        }
        if (wA) todoA = false;
        if (wB) todoB = false;
    }
}

// ---------------------------------------------------------------------------
// WY, step 2: one CTA per head walks the tree level by level; warp per node,
// lane l holds columns l, l + 32, ...  Per node, the path's nodes j are
// visited node side first: running decay ratio G_ij, the dot products
// k_i.k_j and q_i.k_j (fixed butterfly), and the sums of f_j.
// ---------------------------------------------------------------------------
template <int D>
__global__ __launch_bounds__(kTreeThreads) void k_gdn_wy_tree(GdnArgs a) {
    constexpr int P = D / 32;
    __shared__ uint16_t up_s[kGdnMaxNodes][kGdnMaxDepth];
    __shared__ uint8_t dep[kGdnMaxNodes];
    __shared__ int maxdep;
    const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int nw = kTreeThreads / 32;
    if (tid == 0) maxdep = 0;
    __syncthreads();
    for (int i = tid; i < a.n; i += kTreeThreads) {
        const int L = walk_up(a, i, up_s[i]);
        dep[i] = (uint8_t)L;
        if (L > 0) {
            atomicMax(&maxdep, L);
        } else {
            atomicExch(a.err, 1);
            float *out = a.o + ((int64_t)i * a.H + h) * D;
            for (int c = 0; c < D; ++c) out[c] = __int_as_float(0x7FC00000);
        }
    }
    __syncthreads();
    const int md = maxdep;
    const float *G1 = a.G, *G2 = a.G + (int64_t)a.n * a.H * D;
    for (int lev = 1; lev <= md; ++lev) {
        for (int i = warp; i < a.n; i += nw) {
            if (dep[i] != lev) continue;
            const int64_t ih = ((int64_t)i * a.H + h) * D;
            float ki[P], qi[P], facc[P], oacc[P];
#pragma unroll
            for (int m = 0; m < P; ++m) {
                ki[m] = bf2f(a.k[ih + lane + 32 * m]);
                qi[m] = bf2f(a.q[ih + lane + 32 * m]);
                facc[m] = 0.f;
                oacc[m] = 0.f;
            }
            // the ancestors j = up[1..lev-1]; ratio = product of alpha over up[0..s-1]
            float ratio = a.alpha[(int64_t)i * a.H + h];
            for (int s = 1; s < lev; ++s) {
                const int j = up_s[i][s];
                const int64_t jh = ((int64_t)j * a.H + h) * D;
                float pk = 0.f, pq = 0.f, kj[P];
#pragma unroll
                for (int m = 0; m < P; ++m) {
                    kj[m] = bf2f(a.k[jh + lane + 32 * m]);
                    pk = fmaf(ki[m], kj[m], pk);
                    pq = fmaf(qi[m], kj[m], pq);
                }
                const float ck = ratio * warp_sum(pk), cq = ratio * warp_sum(pq);
#pragma unroll
                for (int m = 0; m < P; ++m) {
                    const float fj = a.f[jh + lane + 32 * m];
                    facc[m] = fmaf(ck, fj, facc[m]);
                    oacc[m] = fmaf(cq, fj, oacc[m]);
                }
                ratio *= a.alpha[(int64_t)j * a.H + h];
            }
            const float gamma = ratio;  // alpha over the whole path
            const float be = a.beta[(int64_t)i * a.H + h];
            float pself = 0.f;
#pragma unroll
            for (int m = 0; m < P; ++m) pself = fmaf(qi[m], ki[m], pself);
            const float cself = warp_sum(pself);
            float *out = a.o + ih;
#pragma unroll
            for (int m = 0; m < P; ++m) {
                const int c = lane + 32 * m;
                const float fi = be * (bf2f(a.v[ih + c]) - fmaf(gamma, G1[ih + c], facc[m]));
                a.f[ih + c] = fi;
                out[c] = fmaf(gamma, G2[ih + c], fmaf(cself, fi, oacc[m]));
            }
        }
        __syncthreads();  // this level's f is read by the next
    }
}

template <int D>
cudaError_t launch_gdn_d(const GdnArgs &a, int mode, cudaStream_t s) {
    if (mode == 0) {
        k_gdn_path<D><<<dim3((unsigned)a.n, (unsigned)a.H), 2 * D, 0, s>>>(a);
        return cudaGetLastError();
    }
    k_gdn_proj<D><<<dim3((unsigned)(2 * ((a.n + 15) / 16)), (unsigned)a.H), D, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_gdn_wy_tree<D><<<(unsigned)a.H, kTreeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t gdn_workspace_bytes(int64_t n, int64_t H, int64_t D, int mode) {
    if (mode == 0) return 256;
    return 256 + (size_t)3 * (size_t)n * (size_t)H * (size_t)D * 4;
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
    a.f = a.G + (int64_t)2 * n * H * D;
    if (D == 64) return launch_gdn_d<64>(a, mode, s);
    if (D == 128) return launch_gdn_d<128>(a, mode, s);
    return cudaErrorInvalidValue;
}

}  // namespace w12
