/*
 * w12.h - C ABI of the W12 library (GB300 / sm_103a).
 *
 * W12 is the lossless 12-bit BF16 weight format of "SpecPilot: Autonomous
 * Algorithm Discovery and Systems Optimization for Speculative Decoding"
 * (arXiv 2611.02501), section 4.1: every weight is a sign bit, a 4-bit
 * exponent offset inside a window of 16 binades chosen per output channel,
 * and the 7 BF16 mantissa bits; weights outside the window, zeros and
 * denormals (and, in this library, Inf/NaN) go to an exact escape list.  The
 * same section describes a GEMM that decodes the records in registers and
 * splits its reduction in a fixed order, so that its result is deterministic,
 * and a bit-for-bit check of every decoded tensor at load time.
 *
 * Conventions shared by every call:
 *   - BF16 values travel as uint16_t bit patterns (no CUDA header needed).
 *   - Pointers marked "device" are CUDA device memory owned by the caller;
 *     the library never allocates or frees device memory.
 *   - Calls validate their arguments on the host before any launch and
 *     return a w12_status; on an error nothing has been launched, except
 *     where a call says otherwise.
 *   - Calls are asynchronous on `stream` unless documented as synchronous.
 *     `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - The library holds no state between calls and is thread-safe; two calls
 *     that share a workspace must not run concurrently.
 *
 * Tensor layout (the "packed-record layout"; the paper does not fix one):
 *   Np = N rounded up to 16, Kp = K rounded up to 256.  The 12-bit record of
 *   weight (n,k) is s<<11 | off<<7 | m (off = exponent - base[n]); escaped
 *   and padding slots hold record 0.  The records live in two planes, stored
 *   as tiles of 16 rows x 64 columns, tile (t,c) = (n/16, k/64) at index
 *   t*(Kp/64)+c:
 *     hi plane, 1024 bytes per tile: the top 8 record bits (s|off|m[6:4]).
 *       Row i (0..15), column j (0..63) of a tile is byte
 *       (i/8)*512 + (4*(i%8) + j/16)*16 + j%16.  This plane alone is the
 *       8-bit view nested in W12 (section "(3) two-level verification" of
 *       the paper's news-article page).
 *     lo plane, 512 bytes per tile: the low record nibble (m[3:0]).
 *       Slot L = 4*(i%8) + j/16 owns bytes L*16 .. L*16+15: the first 8 for
 *       row i%8, the next 8 for row i%8+8.  Each group of 8 bytes is two
 *       32-bit little-endian words for columns j%16 = 0..7 and 8..15; inside
 *       a word, column u is the high nibble of byte u (u < 4) or the low
 *       nibble of byte u-4 (u >= 4).
 *   This order hands each lane of a warp exactly the operand fragment of a
 *   16x16 BF16 tensor-core tile with 128-bit loads.
 *   base[n] is the window base exponent of row n (1..239).
 *   Escapes: one 32-bit entry each, key<<16 | raw BF16 bits, grouped by
 *   (row stripe t = n/16, column group g = k/256).  With G = w12_groups(K)
 *   groups per stripe, the entries of (t,g) are esc[esc_ptr[t*G+g] ..
 *   esc_ptr[t*G+g+1]-1], sorted by key; the key of weight (n,k) is
 *   (k%256/64)<<10 | (n%16)<<6 | k%64 (tile, row, column inside the group).
 *   esc_ptr has w12_esc_ptr_len(N,K) = Np/16*G + 1 entries, the last = n_esc.
 *   One coalesced 4-byte load per lane fetches the escapes of a group.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *w12_stream_t;

typedef enum {
    W12_OK = 0,
    W12_ERR_INVALID = -1,     /* bad shape, null pointer, bad stride or option */
    W12_ERR_ALIGN = -2,       /* a buffer or stride breaks the alignment rules */
    W12_ERR_CAPACITY = -3,    /* escape arrays or workspace too small */
    W12_ERR_CUDA = -4,        /* a CUDA runtime call failed */
    W12_ERR_MISMATCH = -5,    /* verify found decoded bits != original bits */
    W12_ERR_TIMEOUT = -6,     /* a bounded device-side wait gave up */
    W12_ERR_CORRUPT = -7,     /* the escape list is malformed */
    W12_ERR_UNSUPPORTED = -8  /* requested path not available for this shape/device */
} w12_status;

/* A W12 tensor.  All pointers are device memory owned by the caller. */
typedef struct {
    int64_t N, K;           /* logical shape of the BF16 tensor [N,K] */
    uint8_t *hi;            /* [w12_hi_bytes(N,K)], 16-byte aligned */
    uint8_t *lo;            /* [w12_lo_bytes(N,K)], 16-byte aligned */
    uint8_t *base;          /* [N] */
    int32_t *esc_ptr;       /* [w12_esc_ptr_len(N,K)] */
    uint32_t *esc;          /* [esc_cap] entries key<<16 | BF16 bits */
    int64_t esc_cap;        /* capacity of esc */
    int64_t n_esc;          /* number of escapes (set by w12_encode) */
} w12_tensor;

/* GEMM kernel paths. */
#define W12_PATH_AUTO 0     /* chosen from M alone */
#define W12_PATH_MMA 1      /* decode in registers + mma.sync, 1 <= M <= 16 */
#define W12_PATH_TC 2       /* tcgen05 / TMEM path, 16 <= M <= 256 */

/* w12_gemm_opts.flags bits.
 * W12_GEMM_OVERLAP_PREVIOUS: the caller promises that the W12 tensor is not
 * being written by work still in flight on `stream`.  The GEMM is then
 * launched as a programmatic dependent launch and starts streaming its
 * weights while the previous kernel on the stream drains; it reads A and
 * writes Y and the workspace only after that kernel has completed.  For
 * back-to-back GEMMs over resident weights (a model's forward pass). */
#define W12_GEMM_OVERLAP_PREVIOUS 1

/* W12_GEMM_NESTED8: multiply by the 8-bit view nested in W12 instead of the
 * exact weights (SpecPilot, section 4.1, and the two-level verification of
 * the news article: a low-precision pass reads "the 8-bit weight view nested
 * in W12").  Only the hi plane is read (1 byte per weight instead of 1.5):
 * an in-window weight becomes (-1)^s * 2^(base+off-127) * (1 + m_hi/8), its
 * top 3 mantissa bits.  The pages do not say what the view holds at an
 * escaped position; this library uses the escape's BF16 bits with the 4 low
 * mantissa bits cleared.  So every weight w is replaced by w & 0xFFF0
 * (truncation toward zero).  Accumulation, rounding and determinism are as
 * for the exact GEMM. */
#define W12_GEMM_NESTED8 2

/* W12_GEMM_SILU_MUL: the fused epilogue of a gated MLP's gate/up GEMM.  The
 * pages do not write the layer out; an exact pass over a dense target streams
 * its gate/up weights, and what the next (down) GEMM reads is silu(g) * u,
 * silu(x) = x / (1 + exp(-x)) (the published SiLU gating).  Row layout: in
 * every stripe s of 16 rows, row 16s+i is the gate row and row 16s+8+i the up
 * row of hidden unit 8s+i (i = 0..7), so N must be a multiple of 16
 * (W12_ERR_INVALID otherwise).  Y is [M, N/2] with ldy >= N/2:
 * Y[m, 8s+i] = BF16(silu(g) * u), g and u the FP32 sums of the two rows as the
 * plain GEMM forms them, silu evaluated in FP32, one rounding to BF16. */
#define W12_GEMM_SILU_MUL 4

/* W12_GEMM_TEST_STALL (tests only): on the tensor-core path (M > 16) one
 * wait of the kernel waits for an event that never comes.  Every wait of the
 * kernel is bounded (about a second), so the wait gives up, the CTA aborts,
 * drains its own copies and MMAs, frees its TMEM and records the failure in
 * the workspace error word: the call completes, Y is unspecified and
 * w12_gemm_workspace_status reports W12_ERR_TIMEOUT.  No effect on the
 * small-M path, which has no waits. */
#define W12_GEMM_TEST_STALL (1 << 30)

/* Options of w12_gemm (NULL = all defaults).  Results are bitwise identical
 * for any max_ctas and with or without W12_GEMM_OVERLAP_PREVIOUS; they depend
 * only on (M, N, K, path, split_k, W12_GEMM_NESTED8).
 *
 * How the work is cut.  Both paths cut a GEMM into work items that are a
 * function of (M, N, K, path, split_k) alone, and every CTA walks items
 * blockIdx.x, blockIdx.x + gridDim.x, ...; the order of every sum is fixed
 * by the items, so the grid (max_ctas, the device's SM count, occupancy)
 * never changes a result.  The automatic cut is sized for W12_PLAN_SMS SMs,
 * the SM count of a GB300: one range of work per resident warp (small-M
 * path) or per SM (balanced tensor-core ranges), and K-chunk splits that fill
 * one or two CTAs per SM.  On a part with another SM count the results stay
 * the same and correct; only the balance of work across SMs changes. */
#define W12_PLAN_SMS 152
typedef struct {
    int32_t max_ctas;       /* 0 = as many as fit; >0 caps the grid on either path (tests) */
    int32_t split_k;        /* 0 = chosen from (M,N,K); >0 forces the split */
    int32_t path;           /* W12_PATH_* */
    int32_t flags;          /* W12_GEMM_* bits; unknown bits are rejected */
} w12_gemm_opts;

/* ---- size queries (host only, no CUDA call) ---- */
int64_t w12_rows_padded(int64_t N);          /* Np */
int64_t w12_cols_padded(int64_t K);          /* Kp */
int64_t w12_hi_bytes(int64_t N, int64_t K);  /* Np*Kp */
int64_t w12_lo_bytes(int64_t N, int64_t K);  /* Np*Kp/2 */
int64_t w12_groups(int64_t K);               /* 256-column groups per stripe: Kp/256 */
int64_t w12_esc_ptr_len(int64_t N, int64_t K);  /* Np/16 * w12_groups(K) + 1 */

/* ---- w12_encode ----  BF16 [N,K] -> W12 (paper section 4.1: window per
 * output channel, records, exact escape list).
 * W: device [N rows, stride ldw elements], ldw >= K.  out: N, K, all
 * pointers and esc_cap filled in by the caller; n_esc is written.
 * Synchronous: two launches on `stream` (the window search, then one
 * cooperative pack launch sized to the blocks the device holds at once, which
 * counts, orders and writes the escapes), then one wait on `stream`; the
 * escape count comes back through a host-mapped pinned word (the library
 * keeps one per encode in flight, for reuse).
 * If the tensor needs more than esc_cap escapes the call returns
 * W12_ERR_CAPACITY with out->n_esc = the number needed; the planes, base and
 * esc_ptr are complete and the first esc_cap escapes are written, so the
 * caller can grow the escape array and call again.  Returns W12_ERR_INVALID
 * if the count would not fit an int32 offset, and W12_ERR_TIMEOUT if a
 * bounded wait inside the pack kernel gave up (about 2 s; the tensor is then
 * unspecified). */
w12_status w12_encode(const uint16_t *W, int64_t ldw, w12_tensor *out, w12_stream_t stream);

/* ---- w12_encode_test_stall ----  Tests only: while `on` is nonzero, every
 * w12_encode of this process makes the first block of its pack kernel skip
 * the first grid barrier, so every block's bounded wait runs out (about 2 s
 * per barrier) and the call returns W12_ERR_TIMEOUT.  Off by default. */
void w12_encode_test_stall(int on);

/* ---- w12_decode ----  W12 -> BF16 [N,K] (paper section 4.1: decode is bit
 * for bit).  W_out: device, stride ldw >= K.  Asynchronous.  For a tensor
 * whose escape list is malformed the output is unspecified (but no access
 * leaves the buffers); use w12_verify_roundtrip to detect that. */
w12_status w12_decode(const w12_tensor *w, uint16_t *W_out, int64_t ldw, w12_stream_t stream);

/* ---- w12_verify_roundtrip ----  load-time check (paper section 4.1: every
 * decoded tensor is checked bit for bit).  Counts the (n,k) whose decoded
 * bits differ from W into *n_mismatch (host pointer).  workspace: device,
 * at least w12_verify_workspace_bytes() bytes, any contents.
 * Synchronous.  Returns W12_OK (0 mismatches), W12_ERR_MISMATCH (>0), or
 * W12_ERR_CORRUPT with *n_mismatch = -1 when the escape list is malformed
 * (offsets not starting at 0, not monotone or not ending at n_esc; a key
 * that is >= 4096 or names a weight outside [N,K]; keys not strictly
 * ascending inside a group). */
size_t w12_verify_workspace_bytes(void);
w12_status w12_verify_roundtrip(const uint16_t *W, int64_t ldw, const w12_tensor *w,
                                int64_t *n_mismatch, void *workspace, size_t ws_bytes,
                                w12_stream_t stream);

/* ---- w12_gemm ----  Y[M,N] = A[M,K] * W^T (paper section 4.1: the GEMM
 * decodes records in registers and splits the reduction in a fixed order).
 * A: device BF16, row stride lda (elements), 16-byte aligned, lda % 8 == 0.
 * Y: device BF16, row stride ldy >= N.  FP32 accumulation; each output is
 * rounded once to BF16 (nearest even).  The summation order depends only on
 * (M, N, K, path, split_k), never on the grid, so results are bitwise
 * reproducible.  workspace: device, at least
 * w12_gemm_workspace_bytes(M,N,K,opts) bytes (256 bytes when no split is
 * needed, else 256 KiB of arrival counters plus the FP32 partials),
 * ZERO-FILLED before its first use.  The counters sit at the same offset for
 * every shape and every successful call leaves them at zero, so one
 * workspace serves any sequence of calls on one stream; after a failed call,
 * zero it again.  Asynchronous.
 * M = 0 or N = 0 is a no-op.  K = 0 writes zeros. */
size_t w12_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, const w12_gemm_opts *opts);
w12_status w12_gemm(const uint16_t *A, int64_t lda, const w12_tensor *w, uint16_t *Y,
                    int64_t ldy, int64_t M, void *workspace, size_t ws_bytes,
                    const w12_gemm_opts *opts, w12_stream_t stream);

/* ---- w12_gemm_noalloc ----  The paper has no counterpart to this call; it
 * exists for callers that cannot allocate device memory: engines that plan
 * all of their device memory at start-up and forbid allocation afterwards,
 * plug-ins that run inside another framework's memory pool, and latency-
 * critical loops where cudaMalloc's implicit device synchronisation would
 * stall other streams.  It computes exactly what w12_gemm computes (same
 * kernels, same split, bitwise the same Y) but takes no workspace: it uses a
 * scratch array of W12_NOALLOC_SCRATCH_BYTES built into the library, which
 * every GPU that loads the library keeps until the process exits.  It calls
 * no allocation routine.
 *   - Shapes and options whose w12_gemm workspace would exceed the scratch
 *     return W12_ERR_CAPACITY.  The automatic plan of every shape with
 *     M <= 16 (the small-M path) fits.  Most automatic tensor-core plans
 *     (M > 16) on large layers do not: their split-K partials need 4.8 MB
 *     (M = 17..32) to 40 MB (M = 256) on the 27B-class layer shapes.  With
 *     split_k = 1 forced, every M <= 256 fits (no partials are needed).
 *   - Options that w12_gemm rejects get the same status here.
 *   - The first call on a device looks up the scratch array's device
 *     address there (loading the library's device code on that device); make
 *     that first call before any stream capture.
 *   - Every call shares the one scratch array and clears its counters and
 *     error word on `stream` before use, so calls that overlap on the GPU
 *     (different streams, or different host threads) race and must not be
 *     issued.
 * Asynchronous on `stream`, like w12_gemm. */
#define W12_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
w12_status w12_gemm_noalloc(const uint16_t *A, int64_t lda, const w12_tensor *w, uint16_t *Y,
                            int64_t ldy, int64_t M, const w12_gemm_opts *opts, w12_stream_t stream);

/* ---- w12_gemm_noalloc_status ----  The paper has no counterpart either.
 * Reads and clears the scratch array's error word on the current device:
 * W12_ERR_TIMEOUT if a bounded wait of the last w12_gemm_noalloc call
 * there gave up (its Y is then unspecified), else W12_OK.  Synchronous on
 * `stream`; call it after the w12_gemm_noalloc call it checks and before the
 * next one, which clears the word. */
w12_status w12_gemm_noalloc_status(w12_stream_t stream);

/* ---- w12_gemm_list ----  Several small-M W12 GEMMs in one persistent
 * launch.  The exact pass of a verify step streams every weight of the
 * target (SpecPilot, section 4.1), and weight reads are 80% of the step
 * (English summary, section 6.1): a layer pass is a chain of GEMMs whose
 * launch boundaries would otherwise each cost a ramp-up and a drain.  Here
 * every warp of one resident grid takes its range of each GEMM in list order
 * (the same cut as w12_gemm, so every Y is bitwise what w12_gemm gives) and
 * starts streaming the next GEMM's weights as soon as its own range is done.
 *   items[i].A, lda, Y, ldy, M: as for w12_gemm (1 <= M <= 16, or M = 0 for
 *     an item that does nothing); items[i].w: host pointer to the tensor.
 *   items[i].after: -1, or the index j < i of an item this one depends on:
 *     its A is read only after item j has written all of its Y (use it when
 *     A is item j's output, or is computed from it).  Items without such a
 *     dependency may overlap.
 *   items[i].flags: 0 or W12_GEMM_SILU_MUL (then Y is [M, N/2]).
 *   opts: max_ctas caps the grid; split_k forces every item's split; path
 *     W12_PATH_AUTO or W12_PATH_MMA (W12_ERR_UNSUPPORTED for a tensor-core
 *     path or an item with M > 16); flags: W12_GEMM_NESTED8 for every item;
 *     W12_GEMM_OVERLAP_PREVIOUS: the launch may start streaming weights
 *     while the previous kernel on the stream drains, as for w12_gemm (its
 *     activations, outputs and workspace are touched only after that kernel
 *     has completed); W12_GEMM_TEST_STALL (tests only) makes the first
 *     item's dependency wait run out.
 *   workspace: device, w12_gemm_list_workspace_bytes(items, n, opts) bytes,
 *     16-byte aligned, zero-filled before its first use; every successful
 *     call leaves it zeroed.
 * Up to W12_LIST_MAX items go into one launch; a longer list is cut into
 * several launches, one after the other on the stream.  Items with K = 0 get
 * Y = 0 before the list's launch starts.  Every dependency wait is bounded
 * (about a second): if one gives up, the call still completes, Y is
 * unspecified and w12_gemm_workspace_status reports W12_ERR_TIMEOUT.  The
 * launch is cooperative (every block resident), which those waits rely on.
 * Asynchronous. */
#define W12_LIST_MAX 64
typedef struct {
    const uint16_t *A;
    int64_t lda;
    const w12_tensor *w;
    uint16_t *Y;
    int64_t ldy;
    int64_t M;
    int32_t after;
    int32_t flags;
} w12_gemm_item;
size_t w12_gemm_list_workspace_bytes(const w12_gemm_item *items, int32_t n, const w12_gemm_opts *opts);
w12_status w12_gemm_list(const w12_gemm_item *items, int32_t n, void *workspace, size_t ws_bytes,
                         const w12_gemm_opts *opts, w12_stream_t stream);

/* Reads (and clears) the device-side error word that bounded waits inside
 * w12_gemm set when they give up.  Synchronous on `stream`.  Returns W12_OK
 * or W12_ERR_TIMEOUT. */
w12_status w12_gemm_workspace_status(void *workspace, size_t ws_bytes, w12_stream_t stream);

/* ---- w12_tree_select ----  Best-first draft-tree node selection: which
 * drafted nodes a verify pass checks (paper: the news-article page's part
 * "(2) best-first tree verification"; the English summary's section 4.4, a
 * node budget shared across requests, and 6.4, best-first trees on an
 * 8-position lattice).
 *   lp: device FP32 [R][D][C], 4-byte aligned: lp[r][d][c] is the drafter's
 *     log-probability of candidate c at position d of request r, given the
 *     prefix before it.  Values must be finite (NaN gives an unspecified
 *     order).
 *   A node is a path (c_0..c_{t-1}) from the root, depth t in 1..D; its
 *   score is the FP32 sum lp[r][0][c_0] + lp[r][1][c_1] + ..., added left to
 *   right.  Nodes are kept best-first in the order: score descending, then
 *   depth, then request, then path (lexicographic on candidate indices).
 *   A child never comes before its parent, so the kept nodes form a tree.
 *   shared = 0: the first `budget` nodes of every request, on its own;
 *   shared = 1: the first `budget` nodes over all requests.
 * Outputs (device, caller-owned), one entry per kept node:
 *   req (int32), depth (int32), path (uint64, 8-byte aligned: candidate
 *   indices, 4 bits per position, position 0 in the lowest bits), score
 *   (float), parent (int32: output index of the parent node, -1 at depth 1).
 *   shared = 1: `budget` entries, filled in the order above; count[0] = the
 *   number kept (less than budget only if the lattices hold fewer nodes).
 *   shared = 0: R segments of `budget` entries, request r's nodes in order
 *   at [r*budget, r*budget + count[r]); count has R entries.
 * workspace: device, w12_tree_workspace_bytes(R, budget) bytes, 16-byte
 * aligned, no initial contents needed.  Limits: 1 <= R <= W12_TREE_MAX_REQUESTS,
 * 1 <= D <= W12_TREE_MAX_DEPTH, 1 <= C <= W12_TREE_MAX_CANDIDATES,
 * 1 <= budget <= W12_TREE_MAX_BUDGET (W12_ERR_INVALID otherwise).
 * Asynchronous. */
#define W12_TREE_MAX_DEPTH 16
#define W12_TREE_MAX_CANDIDATES 16
#define W12_TREE_MAX_BUDGET 256
#define W12_TREE_MAX_REQUESTS 65536
size_t w12_tree_workspace_bytes(int32_t R, int32_t budget);
w12_status w12_tree_select(const float *lp, int32_t R, int32_t D, int32_t C, int32_t budget, int32_t shared,
                           int32_t *req, int32_t *depth, uint64_t *path, float *score, int32_t *parent,
                           int32_t *count, void *workspace, size_t ws_bytes, w12_stream_t stream);

/* ---- w12_gdn_tree ----  Recurrent (Gated DeltaNet) layer outputs for the
 * nodes of draft trees, for tree verification on hybrid models (paper: the
 * news-article page's part "(2)", hybrid models with Gated DeltaNet layers;
 * the English summary's section 4.2 bullet on hybrid targets: each node's
 * state is recomputed from the root state along its root path, and a WY
 * kernel turns the chain of rank-one updates into matrix products on tensor
 * cores, differing from the path kernel only in rounding).
 * The recurrence (the published gated delta rule; the pages name the layer
 * but do not write it out), per head, state S a D x D matrix (row = value
 * index, column = key index): along a root path, node t applies
 *     S <- alpha_t S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 * starting from S0 of the node's request, and the node's output is
 * o = S q_t after its own update.
 *   S0: device FP32 [R][H][D][D], the state before the tree, per request.
 *   q, k, v: device BF16 bits [n][H][D] (keys are normally unit length).
 *   alpha, beta: device FP32 [n][H] (decay and write strength, usually in
 *     (0, 1]).
 *   parent: device int32 [n]: parent[i] in [-1, i) (-1: a child of the root,
 *     i.e. of the request's last accepted token); a root path has at most
 *     W12_GDN_MAX_DEPTH nodes.  The tree-selection call's `parent` output has
 *     this form.
 *   req: device int32 [n] request of each node, in [0, R); a child is in its
 *     parent's request.  NULL: every node in request 0.
 *   o: device FP32 [n][H][D], caller-owned.
 *   mode: W12_GDN_PATH (one CTA per node and head applies the path's updates
 *     one by one) or W12_GDN_WY (one product of all keys and queries with S0
 *     on the tensor cores, then one warp per node and head solves its own
 *     root path's rank-one coefficients).  The two agree up to FP32 rounding;
 *     each is deterministic.
 * workspace: device, w12_gdn_workspace_bytes(n, H, D, mode) bytes, 16-byte
 * aligned, no initial contents needed.  Alignment: S0, q, k, v, o 16 bytes;
 * alpha, beta, parent, req 4 bytes (W12_ERR_ALIGN).  Limits: 0 <= n <=
 * W12_GDN_MAX_NODES, D in {64, 128}, 1 <= H <= 65535, 1 <= R <=
 * W12_GDN_MAX_REQUESTS (W12_ERR_INVALID).
 * A tree that breaks the rules on parent / req / depth is detected on the
 * device: the nodes concerned get NaN outputs and w12_gdn_status reports
 * W12_ERR_INVALID for this call.  Asynchronous. */
#define W12_GDN_PATH 0
#define W12_GDN_WY 1
#define W12_GDN_MAX_DEPTH 16
#define W12_GDN_MAX_NODES 1024
#define W12_GDN_MAX_REQUESTS 65536
size_t w12_gdn_workspace_bytes(int64_t n, int64_t H, int64_t D, int32_t mode);
w12_status w12_gdn_tree(const float *S0, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                        const float *beta, const int32_t *parent, const int32_t *req, int64_t n, int64_t H,
                        int64_t R, int64_t D, float *o, void *workspace, size_t ws_bytes, int32_t mode,
                        w12_stream_t stream);
/* The device-side tree check of the last w12_gdn_tree call on this
 * workspace: W12_OK, or W12_ERR_INVALID if the tree broke a rule.
 * Synchronous on `stream`. */
w12_status w12_gdn_status(void *workspace, size_t ws_bytes, w12_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *w12_status_string(w12_status status);

/* Library version, (major << 16) | minor. */
int32_t w12_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
