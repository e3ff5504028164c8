// Internal launch interface between the C-ABI layer (w12_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "w12.h"

namespace w12 {

// Device view of a W12 tensor (plain pointers, sizes precomputed).
struct TensorView {
    int64_t N, K, Np, Kp, KT;  // KT = Kp / 64 tiles per row stripe
    int64_t G;                 // 256-column groups per stripe
    const uint8_t *hi;
    const uint8_t *lo;
    const uint8_t *base;
    const int32_t *esc_ptr;    // [Np/16*G + 1]
    const uint32_t *esc;       // entries key<<16 | BF16 bits
    int64_t n_esc;
};

__host__ __device__ inline int64_t groups_of(int64_t K) { return (K + 255) / 256; }

// GEMM workspace layout, the same for every shape so that one zeroed
// workspace serves any sequence of calls: [0, 256) error word | arrival
// counters for at most kWsMaxCounters stripes / row tiles (zero between
// calls) | FP32 partials.
constexpr int64_t kWsMaxCounters = 1LL << 16;
constexpr size_t kWsCountersOff = 256;
constexpr size_t kWsPartialsOff = kWsCountersOff + 4 * kWsMaxCounters;

// The small-M path's automatic cut (one range per resident warp of
// W12_PLAN_SMS SMs: 16 warps for M <= 8, 12 for M <= 16) needs at most two
// partial slots per range of 16 rows x 8 or 16 token columns; those plans
// fit the library's built-in scratch (w12_gemm_noalloc).
constexpr size_t kMmaAutoPartialBytesM8 = 2 * 16 * (size_t)W12_PLAN_SMS * 16 * 8 * 4;
constexpr size_t kMmaAutoPartialBytesM16 = 2 * 12 * (size_t)W12_PLAN_SMS * 16 * 16 * 4;
static_assert(kWsPartialsOff + kMmaAutoPartialBytesM8 <= W12_NOALLOC_SCRATCH_BYTES &&
                  kWsPartialsOff + kMmaAutoPartialBytesM16 <= W12_NOALLOC_SCRATCH_BYTES,
              "automatic small-M plans must fit the w12_gemm_noalloc scratch");

// Workspace bytes of w12_gemm for (M, N, K, opts), or the status that
// w12_gemm would return for those options (w12_api.cu).
w12_status gemm_plan_bytes(int64_t M, int64_t N, int64_t K, const w12_gemm_opts *opts, size_t *bytes);

// ---- codec (w12_codec.cu) ----
// a1 - a3: base, esc_ptr (inclusive offsets), planes and the escapes below
// esc_cap; *total (device-visible, e.g. host-mapped) gets esc_ptr[P]: < 0 if
// the total does not fit an int32 offset, or an error code that
// encode_timed_out recognises if a bounded wait gave up.  Not written when
// P == 0.  Two launches: the window search, then the pack.  test_stall
// (tests only): the pack's block 0 skips the first grid barrier, so every
// bounded wait runs out and *total gets the timeout code.
cudaError_t launch_encode(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, uint8_t *base, int32_t *esc_ptr,
                          uint8_t *hi, uint8_t *lo, uint32_t *esc, int64_t esc_cap, int32_t *total,
                          bool test_stall, cudaStream_t s);
bool encode_timed_out(int32_t total);
// a4
cudaError_t launch_decode(const TensorView &t, uint16_t *out, int64_t ldo, cudaStream_t s);
// escape-list structure violations of esc_ptr alone added to *bad (device
// counter): for a tensor without groups, where launch_verify has nothing to
// launch.
cudaError_t launch_check_structure(const TensorView &t, int64_t esc_cap,
                                   unsigned long long *bad, cudaStream_t s);
// a5: mismatches added to *count, escape-list structure violations (offsets
// decreasing, esc_ptr[0] != 0, esc_ptr[P] != n_esc, a key out of range, keys
// not increasing within a group) to *structure_bad (device counters).
cudaError_t launch_verify(const TensorView &t, const uint16_t *W, int64_t ldw, unsigned long long *structure_bad,
                          unsigned long long *count, cudaStream_t s);

// ---- GEMM ----
struct GemmArgs {
    const uint16_t *A;
    int64_t lda;
    uint16_t *Y;
    int64_t ldy;
    int64_t M;
    int split;           // forced split (K-chunks per stripe or row tile), 1 otherwise
    // the work units (small-M path: (stripe, group), u = stripe*G + group;
    // tensor-core path: (row tile, group), u = row_tile*G + group) are cut
    // into segments of seglen units, each segment into `per` contiguous
    // ranges (the first rem of q+1 units, the rest of q); `ranges` in all
    int64_t ranges;
    int seglen, per, q, rem;
    int tc_cps;          // tensor-core path: CTAs per SM of the build (1: 16 decoder warps, 2: 8)
    bool tc_ranges;      // tensor-core path: balanced range cut (else S K-chunks per row tile)
    int max_ctas;        // 0 = occupancy-limited persistent grid
    bool overlap;        // launch as a programmatic dependent of the previous kernel
    bool nested8;        // multiply by the nested 8-bit view (hi plane only, escapes & 0xFFF0)
    bool test_stall;     // tensor-core path: make one bounded wait run out (tests of the timeout path)
    bool silu;           // fused gate/up epilogue: Y[m, 8s+i] = silu(row 16s+i) * (row 16s+8+i)
    float *partials;     // tensor-core path: [S][Mpad][Np] (K-chunks) or [2*ranges][Mpad][128] (ranges);
                         // small-M path: [2*ranges][16][MP] fp32
    int32_t *counters;   // arrival counters per stripe (small-M) or row tile (tensor-core)
    int32_t *error;      // device error word
    uint32_t c28, c16;  // 1<<28, 16: multiplicands the decoder needs at run time
};

// Tensor-core path: tcgen05.mma with TMEM accumulators (M <= 256; partials
// laid out [slots][Mpad][128]).
cudaError_t launch_gemm_tc(const TensorView &t, const GemmArgs &g, cudaStream_t s);
// The scheme, cut and build of the tensor-core path for (M, N, K) and a
// forced split (0 = automatic); returns the bytes of FP32 partials it needs.
int64_t gemm_tc_plan(int64_t M, int64_t N, int64_t K, int split_k, bool counters_ok, GemmArgs &g);
int64_t gemm_tc_pad(int64_t M);

// Gated delta rule along draft-tree root paths (w12_gdn.cu); mode 0 = path
// kernel, 1 = WY.
size_t gdn_workspace_bytes(int64_t n, int64_t H, int64_t D, int mode);
cudaError_t launch_gdn_tree(const float *S0, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *alpha, const float *beta, const int32_t *parent, const int32_t *req,
                            int n, int H, int R, int D, float *o, void *workspace, int mode, cudaStream_t s);

// Best-first draft-tree node selection (w12_tree.cu).
size_t tree_workspace_bytes(int64_t R, int64_t budget);
cudaError_t launch_tree_select(const float *lp, int R, int D, int C, int budget, bool shared, int32_t *req,
                               int32_t *depth, uint64_t *path, float *score, int32_t *parent, int32_t *count,
                               void *workspace, cudaStream_t s);

// A list of small-M GEMMs in one persistent launch (w12_gemm_list).  GEMM
// i uses FP32 slots and arrival counters of slice i % kListSlices; a launch
// holds at most kListMax GEMMs (its descriptors travel as kernel parameters).
constexpr int kListSlices = 4;
constexpr int kListMax = W12_LIST_MAX;
struct ListItem {
    TensorView t;
    GemmArgs g;
    int after;  // index (in this launch) of the GEMM whose completion A waits for; -1: none
};
struct ListParams {
    int n;
    int32_t *done;        // [kListMax] ranges completed per GEMM (zero between launches)
    int32_t *exit_count;  // warps finished (zero between launches)
    int32_t *error;       // workspace error word
    uint32_t c28, c16;
    ListItem item[kListMax];
};
static_assert(sizeof(ListParams) <= 32000, "list descriptors must fit the kernel-parameter space");
// overlap: a programmatic dependent launch (the kernel reads A, Y and the
// workspace only after the previous kernel on the stream has completed).
cudaError_t launch_gemm_mma_list(const ListParams &lp, int nb, bool nested8, int max_ctas, bool overlap,
                                 cudaStream_t s);

// Small-M path: decode in registers + mma.sync m16n8k16 (M <= 16).
cudaError_t launch_gemm_mma(const TensorView &t, const GemmArgs &g, cudaStream_t s);
int64_t gemm_mma_partial_cols(int64_t M);  // MP
// The range cut of the small-M path for (M, N, K) and a forced split (0 =
// automatic): fills ranges / seglen / per / q / rem and returns the number of
// partial slots the cut needs (0 when every stripe lies inside one range).
int64_t gemm_mma_plan(int64_t M, int64_t N, int64_t K, int split_k, bool counters_ok, GemmArgs &g);

}  // namespace w12
