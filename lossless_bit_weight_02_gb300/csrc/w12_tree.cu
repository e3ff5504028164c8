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
// step is a lane scan plus a warp argmax (redux on the score, a shuffle
// tournament only on equal scores).
// Per-request budget: the search writes the output directly.
// Shared budget: a first search keeps K1 = min(budget, 2*ceil(budget/R) + 4)
// nodes per request; every list entry then finds its rank in the total order
// over all lists (k_tree_rank, binary searches in parallel), which is its
// output position, and k_tree_parents maps parent links to ranks.  If a list
// that was cut short could still contribute, a flag is raised and a second
// search / rank / parents pass (which return at once when the flag is clear)
// redoes the work with `budget` nodes per request.
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
constexpr int kWarpsPerBlock = 2;  // static shared memory: 2 x 12.8 KB

// Paths are kept as lexicographic keys: position i in the nibble at bits
// 60-4i.., so that for equal depths the numeric order is the path order.
__device__ __forceinline__ uint64_t lex_put(uint64_t key, int pos, uint32_t v) {
    const int sh = 60 - 4 * pos;
    return (key & ~(0xFull << sh)) | ((uint64_t)v << sh);
}

struct TreeOut {
    int32_t *req, *depth;
    uint64_t *path;
    float *score;
    int32_t *parent, *count;
};

// Order key of a node within a request: the score made an unsigned integer
// that grows with the score (+0 and -0 alike), then depth (smaller first),
// so that "a before b" is k1a > k1b, or k1a == k1b and path key a < b.
__device__ __forceinline__ uint64_t order_k1(float score, int depth) {
    const uint32_t u = __float_as_uint(__fadd_rn(score, 0.0f));  // -0 -> +0
    const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)o << 32) | (uint32_t)(0xFFFF - depth);
}
__device__ __forceinline__ int k1_depth(uint64_t k1) { return 0xFFFF - (int)(k1 & 0xFFFF); }
__device__ __forceinline__ bool before_k(uint64_t k1a, uint64_t ka, uint64_t k1b, uint64_t kb) {
    return k1a > k1b || (k1a == k1b && ka < kb);
}

// The lane holding the warp's first entry in the order, or -1 if no lane
// has one.  Each lane offers its own best (have, k1, key; `tag`, compared
// after k1 and before key, is 0 within one request).
// Fast path: one lane holds the largest score (the high word of k1, never
// 0 for a finite score); otherwise a shuffle tournament on the full keys.
__device__ __forceinline__ int warp_first(bool have, uint64_t k1, int tag, uint64_t key) {
    const uint32_t hi = have ? (uint32_t)(k1 >> 32) : 0u;
    const uint32_t m = __reduce_max_sync(kFull, hi);
    const uint32_t ball = __ballot_sync(kFull, have && hi == m);
    if (ball == 0) return -1;
    if ((ball & (ball - 1)) == 0) return __ffs(ball) - 1;
    bool h = have && hi == m;
    int bl = h ? (int)(threadIdx.x & 31) : -1;
    uint64_t b1 = k1, bk = key;
    int bt = tag;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const int ol = __shfl_xor_sync(kFull, bl, off);
        const uint64_t o1 = __shfl_xor_sync(kFull, b1, off);
        const int ot = __shfl_xor_sync(kFull, bt, off);
        const uint64_t ok = __shfl_xor_sync(kFull, bk, off);
        const bool better = o1 > b1 || (o1 == b1 && (ot < bt || (ot == bt && ok < bk)));
        if (ol >= 0 && (bl < 0 || better)) {
            bl = ol;
            b1 = o1;
            bt = ot;
            bk = ok;
        }
    }
    return bl;
}

// One kept node as the per-request lists store it.
struct TreeNode {
    uint64_t k1;    // order key (score, depth)
    uint64_t key;   // lexicographic path key
    uint64_t path;  // output form of the path
    float score;    // the FP32 sum itself (the order key maps -0 to +0)
    int32_t parent; // index in the same request's list, -1 at depth 1
};

struct Frontier {
    uint64_t k1, key, path;
    float score;
    float pscore;      // the parent's score (unused at depth 1)
    int16_t parent;    // index in the request's list, -1 at depth 1 (budget <= 256)
    int16_t last_rank; // rank of the candidate at the last position
};

struct WarpSmem {
    float cand_lp[kMaxDepth][kMaxCand];  // by rank
    uint8_t cand_idx[kMaxDepth][kMaxCand];
    Frontier f[kSlotsPerLane * 32];
};

// mode 0: per-request budget, output written directly (K = budget);
// mode 1: first search of a shared budget (K = K1, lists of stride `stride`);
// mode 2: second search (K = stride = budget), only when *flag is set.
__global__ __launch_bounds__(32 * kWarpsPerBlock) void k_tree_topk(const float *__restrict__ lp, int R, int D, int C,
                                                                   int K, int stride, int mode,
                                                                   TreeNode *__restrict__ lists,
                                                                   int32_t *__restrict__ counts,
                                                                   int32_t *__restrict__ more, int32_t *flag,
                                                                   TreeOut o) {
    __shared__ WarpSmem sm[kWarpsPerBlock];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarpsPerBlock + warp;
    if (mode == 2 && *(volatile int32_t *)flag == 0) return;  // the first pass was enough
    if (mode == 1 && blockIdx.x == 0 && threadIdx.x == 0) *flag = 0;
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

    if (lane == 0) {
        Frontier e;
        e.score = S.cand_lp[0][0];
        e.k1 = order_k1(e.score, 1);
        e.pscore = 0.f;
        e.parent = -1;
        e.last_rank = 0;
        e.key = lex_put(0, 0, S.cand_idx[0][0]);
        e.path = S.cand_idx[0][0];
        S.f[0] = e;
    }
    __syncwarp();
    TreeNode *out = lists + (int64_t)r * stride;
    const int64_t seg = (int64_t)r * K;  // mode 0: this request's output segment
    int fsize = 1, k = 0;
    for (; k < K && fsize > 0; ++k) {
        // this lane's best frontier entry, then the warp's
        int bi = -1;
        uint64_t b1 = 0, bk = 0;
        for (int i = lane; i < fsize; i += 32) {
            const uint64_t k1 = S.f[i].k1, kk = S.f[i].key;
            if (bi < 0 || before_k(k1, kk, b1, bk)) {
                bi = i;
                b1 = k1;
                bk = kk;
            }
        }
        bi = __shfl_sync(kFull, bi, warp_first(bi >= 0, b1, 0, bk));
        // every lane reads the winner and the last entry, then lanes 0..2
        // write in parallel: the output and the move of the last entry into
        // the winner's slot; the first child; the next sibling.
        const Frontier e = S.f[bi];
        const Frontier last = S.f[fsize - 1];
        const int t = k1_depth(e.k1);  // positions 0 .. t-1 are set
        const bool child = t < D;
        const int nr = e.last_rank + 1;
        const bool sib = nr < C;
        __syncwarp();
        if (lane == 0) {
            if (mode == 0) {
                o.req[seg + k] = r;
                o.depth[seg + k] = t;
                o.path[seg + k] = e.path;
                o.score[seg + k] = e.score;
                o.parent[seg + k] = e.parent < 0 ? -1 : (int32_t)(seg + e.parent);
            } else {
                TreeNode n;
                n.k1 = e.k1;
                n.key = e.key;
                n.path = e.path;
                n.score = e.score;
                n.parent = e.parent;
                out[k] = n;
            }
            if (bi != fsize - 1) S.f[bi] = last;
        } else if ((lane == 1 && child) || (lane == 2 && sib)) {
            // one code path for both successors: lane 1 the first child
            // (rank 0 at position t), lane 2 the next sibling (rank nr at t-1)
            const bool is_child = lane == 1;
            const int pos = is_child ? t : t - 1;
            const int rk = is_child ? 0 : nr;
            const float lpv = S.cand_lp[pos][rk];
            const uint32_t ci = S.cand_idx[pos][rk];
            Frontier x;
            x.pscore = is_child ? e.score : e.pscore;
            x.score = (!is_child && t == 1) ? lpv : __fadd_rn(x.pscore, lpv);
            x.k1 = order_k1(x.score, is_child ? t + 1 : t);
            x.parent = is_child ? (int16_t)k : e.parent;
            x.last_rank = (int16_t)rk;
            x.key = lex_put(e.key, pos, ci);
            x.path = (e.path & ~(0xFull << (4 * pos))) | ((uint64_t)ci << (4 * pos));
            S.f[fsize - 1 + (is_child ? 0 : (child ? 1 : 0))] = x;
        }
        fsize += (child ? 1 : 0) + (sib ? 1 : 0) - 1;
        __syncwarp();
    }
    if (lane == 0) {
        if (mode == 0) {
            o.count[r] = k;
        } else {
            counts[r] = k;
            more[r] = fsize > 0;  // the list was cut short
        }
    }
}

// Shared budget: a node's output position is its rank, the number of list
// entries (over all requests) that come before it in the order (score,
// depth, request, path).  One warp per list entry; lane j binary-searches
// the lists j, j + 32, ... (sorted in the order) for how many of their
// entries come first.  map[r][k] = rank.  If the last entry of a list cut
// short ranks inside the budget, the lists are not long enough: the flag is
// raised and the second pass redoes everything with full lists (entries a
// cut list lacks all come after its last entry, so when that entry ranks
// outside the budget every rank inside it is exact).
__device__ __forceinline__ bool before_r(uint64_t k1a, int ra, uint64_t ka, uint64_t k1b, int rb, uint64_t kb) {
    if (k1a != k1b) return k1a > k1b;
    if (ra != rb) return ra < rb;
    return ka < kb;
}

__global__ __launch_bounds__(256) void k_tree_rank(const TreeNode *__restrict__ lists,
                                                   const int32_t *__restrict__ counts,
                                                   const int32_t *__restrict__ more, int32_t *flag, int pass, int R,
                                                   int K, int budget, int32_t *__restrict__ map, TreeOut o) {
    if (pass == 2 && *(volatile int32_t *)flag == 0) return;
    const int lane = threadIdx.x & 31;
    const int64_t x = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // list entry (warp-uniform)
    if (x >= (int64_t)R * K) return;
    const int r = (int)(x / K), k = (int)(x - (int64_t)r * K);
    if (k >= counts[r]) return;
    const TreeNode n = lists[x];
    int64_t rank = 0;
    for (int q = lane; q < R; q += 32) {
        if (q == r) {
            rank += k;  // its own list is sorted
            continue;
        }
        int lo = 0, hi = counts[q];  // first entry of list q that does not come before n
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const TreeNode &m = lists[(int64_t)q * K + mid];
            if (before_r(m.k1, q, m.key, n.k1, r, n.key))
                lo = mid + 1;
            else
                hi = mid;
        }
        rank += lo;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) rank += __shfl_xor_sync(kFull, rank, off);
    if (lane == 0) {
        map[x] = rank < budget ? (int32_t)rank : -1;
        if (pass == 1 && more[r] && k == counts[r] - 1 && rank < budget) *flag = 1;
        if (rank < budget) {
            o.req[rank] = r;
            o.depth[rank] = k1_depth(n.k1);
            o.path[rank] = n.path;
            o.score[rank] = n.score;
        }
    }
}

// Parents (by their ranks) and the count, once every rank is known.
__global__ __launch_bounds__(256) void k_tree_parents(const TreeNode *__restrict__ lists,
                                                      const int32_t *__restrict__ counts, int32_t *flag, int pass,
                                                      int R, int K, int budget, const int32_t *__restrict__ map,
                                                      TreeOut o) {
    const int f = *(volatile int32_t *)flag;
    if ((pass == 2) != (f != 0)) return;  // pass 1 stands unless the flag is up; then pass 2 does this
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < (int64_t)R * K;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(x / K), k = (int)(x - (int64_t)r * K);
        if (k >= counts[r] || map[x] < 0) continue;
        const int p = lists[x].parent;
        o.parent[map[x]] = p < 0 ? -1 : map[(int64_t)r * K + p];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        int64_t total = 0;
        for (int r = 0; r < R; ++r) total += counts[r];
        *o.count = (int32_t)(total < budget ? total : budget);
    }
}

}  // namespace

size_t tree_workspace_bytes(int64_t R, int64_t budget) {
    // flag | lists [R][budget] | counts, more, (spare) [R] | map [R][budget]
    return 256 + (size_t)R * budget * sizeof(TreeNode) + (size_t)R * 4 * 3 + (size_t)R * budget * 4;
}

cudaError_t launch_tree_select(const float *lp, int R, int D, int C, int budget, bool shared, int32_t *req,
                               int32_t *depth, uint64_t *path, float *score, int32_t *parent, int32_t *count,
                               void *workspace, cudaStream_t s) {
    char *ws = static_cast<char *>(workspace);
    int32_t *flag = reinterpret_cast<int32_t *>(ws);
    TreeNode *lists = reinterpret_cast<TreeNode *>(ws + 256);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + 256 + (size_t)R * budget * sizeof(TreeNode));
    int32_t *more = counts + R;
    int32_t *heads = more + R;
    int32_t *map = heads + R;
    const TreeOut o{req, depth, path, score, parent, count};
    const int blocks = (R + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const dim3 grid(blocks), block(32 * kWarpsPerBlock);
    if (!shared) {
        k_tree_topk<<<grid, block, 0, s>>>(lp, R, D, C, budget, budget, 0, lists, counts, more, flag, o);
        return cudaGetLastError();
    }
    int k1 = 2 * ((budget + R - 1) / R) + 4;
    if (k1 > budget) k1 = budget;
    const int64_t entries = (int64_t)R * budget;
    const unsigned rank_blocks = (unsigned)((entries * 32 + 255) / 256);
    const unsigned fix_blocks = (unsigned)((entries + 255) / 256 < 1024 ? (entries + 255) / 256 : 1024);
    for (int pass = 1; pass <= 2; ++pass) {
        k_tree_topk<<<grid, block, 0, s>>>(lp, R, D, C, pass == 1 ? k1 : budget, budget, pass, lists, counts, more,
                                           flag, o);
        k_tree_rank<<<rank_blocks, 256, 0, s>>>(lists, counts, more, flag, pass, R, budget, budget, map, o);
        k_tree_parents<<<fix_blocks, 256, 0, s>>>(lists, counts, flag, pass, R, budget, budget, map, o);
    }
    return cudaGetLastError();
}

}  // namespace w12
