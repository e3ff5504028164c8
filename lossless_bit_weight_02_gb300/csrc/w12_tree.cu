// Best-first draft-tree node selection (SpecPilot, arXiv 2611.02501: the
// news article's part "(2) best-first tree verification", the English
// summary's section 4.4 (a node budget shared across requests) and 6.4
// (best-first trees on an 8-position lattice)).
//
// Input: per request r a drafter's lattice lp[r][d][c] (FP32 log-probability
// of candidate c at position d given the prefix).  A node is a path of
// candidates from the root; its score is the FP32 left-to-right sum of its
// log-probabilities.  Nodes are kept in the total order (score descending,
// depth, request, path ascending) until the budget is spent; a child never
// precedes its parent in that order, so the kept set is a tree.
//
// k_tree_topk: one warp per request.  The candidates of every position are
// ranked (log-probability descending, index ascending), and the warp runs a
// best-first search whose frontier holds, for every kept node, at most two
// successors: its first child (rank 0 at the next position) and its next
// sibling (the next rank at its own position).  Every node has exactly one
// such predecessor, which precedes it in the order, so popping the best
// frontier entry `budget` times yields the request's first nodes in order.
// The frontier lives in shared memory (at most budget + 1 entries); each
// step is a lane scan plus a shuffle argmax.
// k_tree_merge (shared budget): one warp merges the requests' sorted lists
// in the total order and rewrites parent indices.
#include <cstdint>

#include "w12.h"
#include "w12_device.cuh"
#include "w12_internal.h"

namespace w12 {
namespace {

constexpr int kMaxDepth = W12_TREE_MAX_DEPTH;      // 16: 4-bit path fields in 64 bits
constexpr int kMaxCand = W12_TREE_MAX_CANDIDATES;  // 16
constexpr int kMaxBudget = W12_TREE_MAX_BUDGET;    // 256
constexpr int kSlotsPerLane = (kMaxBudget + 1 + 31) / 32;  // frontier capacity per lane
constexpr int kWarpsPerBlock = 4;

// Paths are kept as lexicographic keys: position i in the nibble at bits
// 60-4i.., so that for equal depths the numeric order is the path order.
__device__ __forceinline__ uint64_t lex_put(uint64_t key, int pos, uint32_t v) {
    const int sh = 60 - 4 * pos;
    return (key & ~(0xFull << sh)) | ((uint64_t)v << sh);
}
__device__ __forceinline__ uint32_t lex_get(uint64_t key, int pos) { return (uint32_t)(key >> (60 - 4 * pos)) & 0xFu; }
// position 0 in the lowest nibble (the output form)
__device__ __forceinline__ uint64_t lex_to_path(uint64_t key) {
    uint64_t p = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) p |= (uint64_t)lex_get(key, i) << (4 * i);
    return p;
}

// One kept node as the per-request lists store it.
struct TreeNode {
    float score;
    int32_t depth;
    int32_t parent;  // index in the same request's list, -1 at depth 1
    int32_t pad;
    uint64_t key;    // lexicographic path key
};

struct Frontier {
    float score, pscore;  // the node's score, its parent's (0 at depth 1)
    int32_t depth, parent;
    uint64_t rank_key;    // ranks, lexicographic layout
    uint64_t key;         // candidate indices, lexicographic layout
};

struct WarpSmem {
    float cand_lp[kMaxDepth][kMaxCand];  // by rank
    uint8_t cand_idx[kMaxDepth][kMaxCand];
    Frontier f[kSlotsPerLane * 32];
};

// true when node a comes before node b in the order (same request)
__device__ __forceinline__ bool before(float sa, int da, uint64_t ka, float sb, int db, uint64_t kb) {
    if (sa != sb) return sa > sb;
    if (da != db) return da < db;
    return ka < kb;
}

__global__ __launch_bounds__(32 * kWarpsPerBlock) void k_tree_topk(const float *__restrict__ lp, int R, int D, int C,
                                                                   int K, TreeNode *__restrict__ lists,
                                                                   int32_t *__restrict__ counts) {
    __shared__ WarpSmem sm[kWarpsPerBlock];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarpsPerBlock + warp;
    if (r >= R) return;  // whole warps only
    WarpSmem &S = sm[warp];
    const float *L = lp + (int64_t)r * D * C;

    // rank the candidates of every position: log-probability descending,
    // index ascending
    for (int x = lane; x < D * C; x += 32) {
        const int d = x / C, c = x - d * C;
        const float v = L[x];
        int rank = 0;
        for (int j = 0; j < C; ++j) {
            const float u = L[d * C + j];
            rank += (u > v || (u == v && j < c)) ? 1 : 0;
        }
        S.cand_lp[d][rank] = v;
        S.cand_idx[d][rank] = (uint8_t)c;
    }
    __syncwarp();

    int fsize = 1;
    if (lane == 0) {
        Frontier e;
        e.score = S.cand_lp[0][0];
        e.pscore = 0.f;
        e.depth = 1;
        e.parent = -1;
        e.rank_key = 0;
        e.key = lex_put(0, 0, S.cand_idx[0][0]);
        S.f[0] = e;
    }
    __syncwarp();
    TreeNode *out = lists + (int64_t)r * K;
    int k = 0;
    for (; k < K && fsize > 0; ++k) {
        // the best frontier entry: lane scan, then a shuffle argmax
        int bi = -1;
        float bs = 0.f;
        int bd = 0;
        uint64_t bk = 0;
        for (int j = 0; j < kSlotsPerLane; ++j) {
            const int i = lane + 32 * j;
            if (i < fsize) {
                const Frontier &e = S.f[i];
                if (bi < 0 || before(e.score, e.depth, e.key, bs, bd, bk)) {
                    bi = i;
                    bs = e.score;
                    bd = e.depth;
                    bk = e.key;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const int oi = __shfl_xor_sync(kFull, bi, off);
            const float os = __shfl_xor_sync(kFull, bs, off);
            const int od = __shfl_xor_sync(kFull, bd, off);
            const uint64_t ok = __shfl_xor_sync(kFull, bk, off);
            if (oi >= 0 && (bi < 0 || before(os, od, ok, bs, bd, bk))) {
                bi = oi;
                bs = os;
                bd = od;
                bk = ok;
            }
        }
        // every lane holds the same winner
        if (lane == 0) {
            const Frontier e = S.f[bi];
            TreeNode n;
            n.score = e.score;
            n.depth = e.depth;
            n.parent = e.parent;
            n.pad = 0;
            n.key = e.key;
            out[k] = n;
            // remove it, then add its first child and its next sibling
            int sz = fsize - 1;
            S.f[bi] = S.f[sz];
            const int t = e.depth;  // positions 0 .. t-1 are set
            if (t < D) {
                Frontier c;
                c.pscore = e.score;
                c.score = __fadd_rn(e.score, S.cand_lp[t][0]);
                c.depth = t + 1;
                c.parent = k;
                c.rank_key = lex_put(e.rank_key, t, 0);
                c.key = lex_put(e.key, t, S.cand_idx[t][0]);
                S.f[sz++] = c;
            }
            const uint32_t nr = lex_get(e.rank_key, t - 1) + 1;
            if ((int)nr < C) {
                Frontier s;
                s.pscore = e.pscore;
                s.score = t == 1 ? S.cand_lp[0][nr] : __fadd_rn(e.pscore, S.cand_lp[t - 1][nr]);
                s.depth = t;
                s.parent = e.parent;
                s.rank_key = lex_put(e.rank_key, t - 1, nr);
                s.key = lex_put(e.key, t - 1, S.cand_idx[t - 1][nr]);
                S.f[sz++] = s;
            }
            fsize = sz;
        }
        fsize = __shfl_sync(kFull, fsize, 0);
        __syncwarp();
    }
    if (lane == 0) counts[r] = k;
}

// Per-request budget: the lists become the output, request after request in
// segments of `budget` entries, parents as indices into the whole output.
__global__ void k_tree_emit(const TreeNode *__restrict__ lists, const int32_t *__restrict__ counts, int R, int K,
                            int32_t *req, int32_t *depth, uint64_t *path, float *score, int32_t *parent,
                            int32_t *count) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= (int64_t)R * K) return;
    const int r = (int)(x / K), i = (int)(x - (int64_t)r * K);
    if (i == 0) count[r] = counts[r];
    if (i >= counts[r]) return;
    const TreeNode n = lists[x];
    req[x] = r;
    depth[x] = n.depth;
    path[x] = lex_to_path(n.key);
    score[x] = n.score;
    parent[x] = n.parent < 0 ? -1 : (int32_t)((int64_t)r * K + n.parent);
}

// Shared budget: `budget` steps of a warp argmax over the requests' list
// heads in the total order (the request is the third key).  map[r][i] is
// the output index of list entry i of request r; a parent is emitted before
// its children.
__device__ __forceinline__ bool before_r(float sa, int da, int ra, uint64_t ka, float sb, int db, int rb,
                                         uint64_t kb) {
    if (sa != sb) return sa > sb;
    if (da != db) return da < db;
    if (ra != rb) return ra < rb;
    return ka < kb;
}

__global__ __launch_bounds__(32) void k_tree_merge(const TreeNode *__restrict__ lists,
                                                   const int32_t *__restrict__ counts, int R, int K, int budget,
                                                   int32_t *__restrict__ heads, int32_t *__restrict__ map,
                                                   int32_t *req, int32_t *depth, uint64_t *path, float *score,
                                                   int32_t *parent, int32_t *count) {
    const int lane = threadIdx.x;
    for (int r = lane; r < R; r += 32) heads[r] = 0;
    __syncwarp();
    int n_out = 0;
    for (; n_out < budget; ++n_out) {
        int br = -1;
        float bs = 0.f;
        int bd = 0;
        uint64_t bk = 0;
        for (int r = lane; r < R; r += 32) {
            const int h = heads[r];
            if (h < counts[r]) {
                const TreeNode &n = lists[(int64_t)r * K + h];
                if (br < 0 || before_r(n.score, n.depth, r, n.key, bs, bd, br, bk)) {
                    br = r;
                    bs = n.score;
                    bd = n.depth;
                    bk = n.key;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const int orr = __shfl_xor_sync(kFull, br, off);
            const float os = __shfl_xor_sync(kFull, bs, off);
            const int od = __shfl_xor_sync(kFull, bd, off);
            const uint64_t ok = __shfl_xor_sync(kFull, bk, off);
            if (orr >= 0 && (br < 0 || before_r(os, od, orr, ok, bs, bd, br, bk))) {
                br = orr;
                bs = os;
                bd = od;
                bk = ok;
            }
        }
        if (br < 0) break;  // every list is exhausted (warp-uniform)
        if (lane == 0) {
            const int h = heads[br];
            const TreeNode n = lists[(int64_t)br * K + h];
            req[n_out] = br;
            depth[n_out] = n.depth;
            path[n_out] = lex_to_path(n.key);
            score[n_out] = n.score;
            parent[n_out] = n.parent < 0 ? -1 : map[(int64_t)br * K + n.parent];
            map[(int64_t)br * K + h] = n_out;
            heads[br] = h + 1;
        }
        __syncwarp();
    }
    if (lane == 0) *count = n_out;
}

}  // namespace

size_t tree_workspace_bytes(int64_t R, int64_t budget) {
    const size_t lists = (size_t)R * budget * sizeof(TreeNode);
    return 256 + lists + (size_t)R * 4 * 2 + (size_t)R * budget * 4;
}

cudaError_t launch_tree_select(const float *lp, int R, int D, int C, int budget, bool shared, int32_t *req,
                               int32_t *depth, uint64_t *path, float *score, int32_t *parent, int32_t *count,
                               void *workspace, cudaStream_t s) {
    char *ws = static_cast<char *>(workspace);
    TreeNode *lists = reinterpret_cast<TreeNode *>(ws + 256);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + 256 + (size_t)R * budget * sizeof(TreeNode));
    int32_t *heads = counts + R;
    int32_t *map = heads + R;
    const int blocks = (R + kWarpsPerBlock - 1) / kWarpsPerBlock;
    k_tree_topk<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(lp, R, D, C, budget, lists, counts);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (shared) {
        k_tree_merge<<<1, 32, 0, s>>>(lists, counts, R, budget, budget, heads, map, req, depth, path, score, parent,
                                      count);
    } else {
        const int64_t n = (int64_t)R * budget;
        k_tree_emit<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(lists, counts, R, budget, req, depth, path, score,
                                                                 parent, count);
    }
    return cudaGetLastError();
}

}  // namespace w12
