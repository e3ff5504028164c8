// C-ABI layer of the W12 library: argument validation, workspace layout and
// kernel launches.  Every public entry point is declared in include/w12.h.
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "w12.h"
#include "w12_device.cuh"
#include "w12_internal.h"

namespace {

using namespace w12;

constexpr int64_t kMaxK = (1LL << 31) - 128;  // columns are int32 in the escape list
constexpr int64_t kMaxN = 1LL << 30;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

w12_status check_tensor(const w12_tensor *w) {
    if (!w) return W12_ERR_INVALID;
    if (w->N < 0 || w->K < 0 || w->N > kMaxN || w->K > kMaxK) return W12_ERR_INVALID;
    if (w->esc_cap < 0 || w->n_esc < 0) return W12_ERR_INVALID;
    if (!w->esc_ptr) return W12_ERR_INVALID;
    if (w->N > 0 && !w->base) return W12_ERR_INVALID;
    if (w->N > 0 && w->K > 0) {
        if (!w->hi || !w->lo) return W12_ERR_INVALID;
        if (!aligned16(w->hi) || !aligned16(w->lo)) return W12_ERR_ALIGN;
    }
    if (w->esc_cap > 0 && !w->esc) return W12_ERR_INVALID;
    return W12_OK;
}

TensorView view_of(const w12_tensor *w) {
    TensorView t;
    t.N = w->N;
    t.K = w->K;
    t.Np = rows_padded(w->N);
    t.Kp = cols_padded(w->K);
    t.KT = t.Kp / 64;
    t.G = groups_of(w->K);
    t.hi = w->hi;
    t.lo = w->lo;
    t.base = w->base;
    t.esc_ptr = w->esc_ptr;
    t.esc = w->esc;
    t.n_esc = w->n_esc < w->esc_cap ? w->n_esc : w->esc_cap;
    return t;
}

struct GemmPlan {
    int path;
    int split;
    GemmArgs cut{};  // small-M path range cut
    int64_t mp;  // partial columns
    size_t counters_off, partials_off, bytes;
};

int choose_path(int64_t M, const w12_gemm_opts *o) {
    const int p = o ? o->path : W12_PATH_AUTO;
    if (p != W12_PATH_AUTO) return p;
    return M <= 16 ? W12_PATH_MMA : W12_PATH_TC;
}

w12_status plan_gemm(int64_t M, int64_t N, int64_t K, const w12_gemm_opts *o, GemmPlan &pl) {
    if (M < 0 || N < 0 || K < 0 || N > kMaxN || K > kMaxK) return W12_ERR_INVALID;
    if (o && ((o->flags & ~(W12_GEMM_OVERLAP_PREVIOUS | W12_GEMM_NESTED8 | W12_GEMM_TEST_STALL |
                            W12_GEMM_SILU_MUL)) != 0 ||
              o->max_ctas < 0 || o->split_k < 0 ||
              o->split_k > 256))
        return W12_ERR_INVALID;
    pl.path = choose_path(M, o);
    if (pl.path != W12_PATH_MMA && pl.path != W12_PATH_TC) return W12_ERR_INVALID;
    if (pl.path == W12_PATH_MMA && M > 16) return W12_ERR_UNSUPPORTED;
    if (pl.path == W12_PATH_TC && M > 256) return W12_ERR_UNSUPPORTED;
    const bool tc = pl.path == W12_PATH_TC;
    const int64_t G = groups_of(K);
    const int64_t Np = rows_padded(N);
    const bool counters_ok = Np / 16 <= kWsMaxCounters;  // arrival counters exist for at most kWsMaxCounters stripes
    // Fixed layout, the same for every shape, so that the counter region is
    // never reused for partials (w12_internal.h).
    pl.counters_off = kWsCountersOff;
    pl.partials_off = kWsPartialsOff;
    if (tc) {
        pl.mp = gemm_tc_pad(M);
        const int64_t pbytes = gemm_tc_plan(M, N, K, o ? o->split_k : 0, counters_ok, pl.cut);
        pl.split = pl.cut.split;
        pl.bytes = pbytes > 0 ? pl.partials_off + (size_t)pbytes : 256;
    } else {
        // The kernel indexes a lane's hi-plane bytes with 256 * unit + lane in
        // 32 bits: at most 2^24 (stripe, group) units, 64 GiB of hi plane.
        if (Np / 16 * G >= (1LL << 24)) return W12_ERR_INVALID;
        pl.split = 1;
        pl.mp = gemm_mma_partial_cols(M);
        const int64_t slots = gemm_mma_plan(M, N, K, o ? o->split_k : 0, counters_ok, pl.cut);
        pl.bytes = slots > 0 ? pl.partials_off + (size_t)slots * 16 * pl.mp * 4 : 256;
    }
    return W12_OK;
}

w12_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W12_OK : W12_ERR_CUDA; }

}  // namespace

namespace w12 {
w12_status gemm_plan_bytes(int64_t M, int64_t N, int64_t K, const w12_gemm_opts *opts, size_t *bytes) {
    GemmPlan pl;
    const w12_status st = plan_gemm(M, N, K, opts, pl);
    *bytes = st == W12_OK ? pl.bytes : 0;
    return st;
}
}  // namespace w12

extern "C" {

int64_t w12_rows_padded(int64_t N) { return N < 0 ? -1 : rows_padded(N); }
int64_t w12_cols_padded(int64_t K) { return K < 0 ? -1 : cols_padded(K); }
int64_t w12_hi_bytes(int64_t N, int64_t K) { return (N < 0 || K < 0) ? -1 : rows_padded(N) * cols_padded(K); }
int64_t w12_lo_bytes(int64_t N, int64_t K) {
    return (N < 0 || K < 0) ? -1 : rows_padded(N) * cols_padded(K) / 2;
}

int64_t w12_groups(int64_t K) { return K < 0 ? -1 : groups_of(K); }
int64_t w12_esc_ptr_len(int64_t N, int64_t K) {
    return (N < 0 || K < 0) ? -1 : rows_padded(N) / 16 * groups_of(K) + 1;
}

int32_t w12_version(void) { return (1 << 16) | 0; }

const char *w12_status_string(w12_status s) {
    switch (s) {
        case W12_OK: return "W12_OK";
        case W12_ERR_INVALID: return "W12_ERR_INVALID";
        case W12_ERR_ALIGN: return "W12_ERR_ALIGN";
        case W12_ERR_CAPACITY: return "W12_ERR_CAPACITY";
        case W12_ERR_CUDA: return "W12_ERR_CUDA";
        case W12_ERR_MISMATCH: return "W12_ERR_MISMATCH";
        case W12_ERR_TIMEOUT: return "W12_ERR_TIMEOUT";
        case W12_ERR_CORRUPT: return "W12_ERR_CORRUPT";
        case W12_ERR_UNSUPPORTED: return "W12_ERR_UNSUPPORTED";
    }
    return "W12_ERR_UNKNOWN";
}

// Host-mapped words that the pack kernel writes the escape total into, so an
// encode reads it after the stream sync without a copy; one per encode in
// flight (several host threads may encode at once), kept for reuse.
namespace {
class TotalSlots {
  public:
    int32_t *take() {
        {
            std::lock_guard<std::mutex> lock(m_);
            if (!free_.empty()) {
                int32_t *p = free_.back();
                free_.pop_back();
                return p;
            }
        }
        void *p = nullptr;
        if (cudaHostAlloc(&p, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) return nullptr;
        return static_cast<int32_t *>(p);
    }
    void give(int32_t *p) {
        std::lock_guard<std::mutex> lock(m_);
        free_.push_back(p);
    }

  private:
    std::mutex m_;
    std::vector<int32_t *> free_;
};
TotalSlots g_total_slots;
std::atomic<int> g_encode_test_stall{0};

struct SlotGuard {
    int32_t *p;
    ~SlotGuard() {
        if (p) g_total_slots.give(p);
    }
};
}  // namespace

w12_status w12_encode(const uint16_t *W, int64_t ldw, w12_tensor *out, w12_stream_t stream) {
    w12_status st = check_tensor(out);
    if (st != W12_OK) return st;
    if (ldw < out->K) return W12_ERR_INVALID;
    if (out->N > 0 && out->K > 0 && !W) return W12_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t N = out->N, K = out->K;
    const int64_t P = rows_padded(N) / 16 * groups_of(K);  // (stripe, group) count
    // the kernel writes only the entries below esc_cap (none if the offsets
    // overflowed), so the escape total is read once, at the end
    SlotGuard slot{g_total_slots.take()};
    int32_t *dslot = nullptr;
    if (!slot.p || cudaHostGetDevicePointer(reinterpret_cast<void **>(&dslot), slot.p, 0) != cudaSuccess)
        return W12_ERR_CUDA;
    if (launch_encode(W, ldw, N, K, out->base, out->esc_ptr, out->hi, out->lo, out->esc, out->esc_cap, dslot,
                      g_encode_test_stall.load() != 0, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    const int32_t total = P == 0 ? 0 : *reinterpret_cast<volatile int32_t *>(slot.p);
    if (encode_timed_out(total)) return W12_ERR_TIMEOUT;
    if (total < 0) return W12_ERR_INVALID;  // more escapes than an int32 offset can index
    out->n_esc = total;
    return total > out->esc_cap ? W12_ERR_CAPACITY : W12_OK;
}

void w12_encode_test_stall(int on) { g_encode_test_stall.store(on != 0 ? 1 : 0); }

w12_status w12_decode(const w12_tensor *w, uint16_t *W_out, int64_t ldw, w12_stream_t stream) {
    w12_status st = check_tensor(w);
    if (st != W12_OK) return st;
    if (ldw < w->K) return W12_ERR_INVALID;
    if (w->N > 0 && w->K > 0 && !W_out) return W12_ERR_INVALID;
    if (w->N == 0 || w->K == 0) return W12_OK;
    return cuda_status(launch_decode(view_of(w), W_out, ldw, reinterpret_cast<cudaStream_t>(stream)));
}

size_t w12_verify_workspace_bytes(void) { return 16; }

w12_status w12_verify_roundtrip(const uint16_t *W, int64_t ldw, const w12_tensor *w, int64_t *n_mismatch,
                                void *workspace, size_t ws_bytes, w12_stream_t stream) {
    w12_status st = check_tensor(w);
    if (st != W12_OK) return st;
    if (!n_mismatch || ldw < w->K) return W12_ERR_INVALID;
    if (!workspace || ws_bytes < w12_verify_workspace_bytes()) return W12_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(workspace) & 7) return W12_ERR_ALIGN;
    if (w->N > 0 && w->K > 0 && !W) return W12_ERR_INVALID;
    *n_mismatch = -1;
    if (w->n_esc > w->esc_cap) return W12_ERR_CORRUPT;
    if (w->N == 0) {
        *n_mismatch = 0;
        return w->n_esc == 0 ? W12_OK : W12_ERR_CORRUPT;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long *cnt = static_cast<unsigned long long *>(workspace);
    const TensorView t = view_of(w);
    if (cudaMemsetAsync(cnt, 0, 16, s) != cudaSuccess) return W12_ERR_CUDA;
    // one launch checks the escape list's structure and compares every weight
    // (a tensor without columns has only esc_ptr[0] to check)
    if ((w->K > 0 ? launch_verify(t, W, ldw, cnt, cnt + 1, s) : launch_check_structure(t, w->esc_cap, cnt, s)) !=
        cudaSuccess)
        return W12_ERR_CUDA;
    unsigned long long host[2] = {0, 0};
    if (cudaMemcpyAsync(host, cnt, 16, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    if (host[0] != 0) return W12_ERR_CORRUPT;
    *n_mismatch = (int64_t)host[1];
    return host[1] ? W12_ERR_MISMATCH : W12_OK;
}

size_t w12_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, const w12_gemm_opts *opts) {
    GemmPlan pl;
    if (plan_gemm(M, N, K, opts, pl) != W12_OK) return 0;
    return pl.bytes;
}

w12_status w12_gemm(const uint16_t *A, int64_t lda, const w12_tensor *w, uint16_t *Y, int64_t ldy, int64_t M,
                    void *workspace, size_t ws_bytes, const w12_gemm_opts *opts, w12_stream_t stream) {
    w12_status st = check_tensor(w);
    if (st != W12_OK) return st;
    if (M < 0) return W12_ERR_INVALID;
    if (M == 0 || w->N == 0) return W12_OK;
    const bool silu = opts && (opts->flags & W12_GEMM_SILU_MUL) != 0;
    if (silu && w->N % 16 != 0) return W12_ERR_INVALID;
    if (!Y || ldy < (silu ? w->N / 2 : w->N)) return W12_ERR_INVALID;
    if (w->K > 0) {
        if (!A || lda < w->K) return W12_ERR_INVALID;
        if (!aligned16(A) || (lda % 8) != 0) return W12_ERR_ALIGN;
    }
    GemmPlan pl;
    st = plan_gemm(M, w->N, w->K, opts, pl);
    if (st != W12_OK) return st;
    if (w->K == 0)  // empty reduction: Y = 0 (silu(0) * 0 = 0 too)
        return cuda_status(cudaMemset2DAsync(Y, (size_t)ldy * 2, 0, (size_t)(silu ? w->N / 2 : w->N) * 2,
                                             (size_t)M, reinterpret_cast<cudaStream_t>(stream)));
    if (!workspace || ws_bytes < pl.bytes) return W12_ERR_CAPACITY;
    if (!aligned16(workspace)) return W12_ERR_ALIGN;
    char *ws = static_cast<char *>(workspace);
    GemmArgs g;
    g.A = A;
    g.lda = lda;
    g.Y = Y;
    g.ldy = ldy;
    g.M = M;
    g.split = pl.split;
    g.ranges = pl.cut.ranges;
    g.seglen = pl.cut.seglen;
    g.per = pl.cut.per;
    g.q = pl.cut.q;
    g.rem = pl.cut.rem;
    g.tc_cps = pl.cut.tc_cps;
    g.tc_ranges = pl.cut.tc_ranges;
    g.max_ctas = opts ? opts->max_ctas : 0;
    g.overlap = opts ? (opts->flags & W12_GEMM_OVERLAP_PREVIOUS) != 0 : false;
    g.nested8 = opts ? (opts->flags & W12_GEMM_NESTED8) != 0 : false;
    g.test_stall = opts ? (opts->flags & W12_GEMM_TEST_STALL) != 0 : false;
    g.silu = silu;
    g.error = reinterpret_cast<int32_t *>(ws);
    g.counters = reinterpret_cast<int32_t *>(ws + pl.counters_off);
    g.partials = reinterpret_cast<float *>(ws + pl.partials_off);
    g.c28 = 1u << 28;
    g.c16 = 16u;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.path == W12_PATH_TC) {
        const cudaError_t e = launch_gemm_tc(view_of(w), g, s);
        return e == cudaErrorNotSupported ? W12_ERR_UNSUPPORTED : cuda_status(e);
    }
    return cuda_status(launch_gemm_mma(view_of(w), g, s));
}

// ---- w12_gemm_list ----
// Workspace: [0,256) error word | kListSlices slices of arrival counters
// (kWsMaxCounters each) | done[kListMax] + exit counter (256-byte aligned) |
// kListSlices slices of FP32 partials.
namespace {

constexpr size_t kListCountersOff = 256;
constexpr size_t kListDoneOff = kListCountersOff + 4 * (size_t)kListSlices * kWsMaxCounters;
constexpr size_t kListPartialsOff = kListDoneOff + (4 * (kListMax + 1) + 255) / 256 * 256;

// Checks every item and computes the bytes of one partial slice (the largest
// over the list's launches).  Returns the status w12_gemm_list returns.
w12_status plan_list(const w12_gemm_item *items, int32_t n, const w12_gemm_opts *o, size_t *slice_bytes) {
    if (n < 0 || (n > 0 && !items)) return W12_ERR_INVALID;
    if (o && ((o->flags & ~(W12_GEMM_OVERLAP_PREVIOUS | W12_GEMM_NESTED8 | W12_GEMM_TEST_STALL)) != 0 ||
              o->max_ctas < 0 || o->split_k < 0 || o->split_k > 256))
        return W12_ERR_INVALID;
    if (o && o->path != W12_PATH_AUTO && o->path != W12_PATH_MMA)
        return o->path == W12_PATH_TC ? W12_ERR_UNSUPPORTED : W12_ERR_INVALID;
    size_t slice = 0;
    for (int32_t c0 = 0; c0 < n; c0 += kListMax) {
        const int32_t c1 = n - c0 < kListMax ? n : c0 + kListMax;
        int64_t mmax = 0;
        for (int32_t i = c0; i < c1; ++i) mmax = items[i].M > mmax ? items[i].M : mmax;
        const int64_t mp = mmax <= 8 ? 8 : 16;
        for (int32_t i = c0; i < c1; ++i) {
            const w12_gemm_item &it = items[i];
            w12_status st = check_tensor(it.w);
            if (st != W12_OK) return st;
            if (it.M < 0) return W12_ERR_INVALID;
            if (it.M > 16) return W12_ERR_UNSUPPORTED;
            if (it.after < -1 || it.after >= i) return W12_ERR_INVALID;
            if ((it.flags & ~W12_GEMM_SILU_MUL) != 0) return W12_ERR_INVALID;
            const bool silu = (it.flags & W12_GEMM_SILU_MUL) != 0;
            const int64_t N = it.w->N, K = it.w->K;
            if (it.M == 0 || N == 0) continue;
            if (silu && N % 16 != 0) return W12_ERR_INVALID;
            if (!it.Y || it.ldy < (silu ? N / 2 : N)) return W12_ERR_INVALID;
            if (K > 0) {
                if (!it.A || it.lda < K) return W12_ERR_INVALID;
                if (!aligned16(it.A) || (it.lda % 8) != 0) return W12_ERR_ALIGN;
            }
            const int64_t G = groups_of(K), Np = rows_padded(N);
            if (Np / 16 * G >= (1LL << 24)) return W12_ERR_INVALID;  // as for w12_gemm's small-M path
            GemmArgs cut{};
            const int64_t slots = gemm_mma_plan(it.M, N, K, o ? o->split_k : 0, Np / 16 <= kWsMaxCounters, cut);
            const size_t b = (size_t)slots * 16 * (size_t)mp * 4;
            slice = b > slice ? b : slice;
        }
    }
    *slice_bytes = (slice + 255) / 256 * 256;
    return W12_OK;
}

}  // namespace

size_t w12_gemm_list_workspace_bytes(const w12_gemm_item *items, int32_t n, const w12_gemm_opts *opts) {
    size_t slice = 0;
    if (plan_list(items, n, opts, &slice) != W12_OK) return 0;
    return kListPartialsOff + (size_t)kListSlices * slice;
}

w12_status w12_gemm_list(const w12_gemm_item *items, int32_t n, void *workspace, size_t ws_bytes,
                         const w12_gemm_opts *opts, w12_stream_t stream) {
    size_t slice = 0;
    w12_status st = plan_list(items, n, opts, &slice);
    if (st != W12_OK) return st;
    if (n == 0) return W12_OK;
    if (!workspace || ws_bytes < kListPartialsOff + (size_t)kListSlices * slice) return W12_ERR_CAPACITY;
    if (!aligned16(workspace)) return W12_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const bool nested8 = opts && (opts->flags & W12_GEMM_NESTED8) != 0;
    const bool stall = opts && (opts->flags & W12_GEMM_TEST_STALL) != 0;
    const bool overlap = opts && (opts->flags & W12_GEMM_OVERLAP_PREVIOUS) != 0;
    static thread_local ListParams lp;  // 15 KB of descriptors: not on the stack
    for (int32_t c0 = 0; c0 < n; c0 += kListMax) {
        const int32_t c1 = n - c0 < kListMax ? n : c0 + kListMax;
        memset(&lp, 0, sizeof lp);
        lp.n = c1 - c0;
        lp.done = reinterpret_cast<int32_t *>(ws + kListDoneOff);
        lp.exit_count = lp.done + kListMax;
        lp.error = reinterpret_cast<int32_t *>(ws);
        lp.c28 = 1u << 28;
        lp.c16 = 16u;
        int64_t mmax = 0;
        bool work = false;
        for (int32_t i = c0; i < c1; ++i) {
            const w12_gemm_item &it = items[i];
            const int j = i - c0;
            ListItem &li = lp.item[j];
            li.t = view_of(it.w);
            li.after = it.after >= c0 ? it.after - c0 : -1;  // earlier launches have completed
            GemmArgs &g = li.g;
            g.ranges = 0;  // no work unless set below
            g.seglen = g.per = g.q = 1;
            const bool silu = (it.flags & W12_GEMM_SILU_MUL) != 0;
            if (it.M == 0 || it.w->N == 0) continue;
            if (it.w->K == 0) {  // empty reduction: Y = 0 before the launch
                if (cudaMemset2DAsync(it.Y, (size_t)it.ldy * 2, 0, (size_t)(silu ? it.w->N / 2 : it.w->N) * 2,
                                      (size_t)it.M, s) != cudaSuccess)
                    return W12_ERR_CUDA;
                continue;
            }
            const int64_t Np = rows_padded(it.w->N);
            (void)gemm_mma_plan(it.M, it.w->N, it.w->K, opts ? opts->split_k : 0, Np / 16 <= kWsMaxCounters, g);
            g.A = it.A;
            g.lda = it.lda;
            g.Y = it.Y;
            g.ldy = it.ldy;
            g.M = it.M;
            g.split = 1;
            g.nested8 = nested8;
            g.silu = silu;
            g.partials = reinterpret_cast<float *>(ws + kListPartialsOff + (size_t)(j % kListSlices) * slice);
            g.counters = reinterpret_cast<int32_t *>(ws + kListCountersOff) + (size_t)(j % kListSlices) * kWsMaxCounters;
            g.error = lp.error;
            g.c28 = lp.c28;
            g.c16 = lp.c16;
            mmax = it.M > mmax ? it.M : mmax;
            work = true;
        }
        // tests only: the first item waits for a count that cannot be reached
        // while it is waiting (every warp's exit), so the wait runs out
        if (stall && c0 == 0) lp.item[0].after = -2;
        if (!work) continue;
        const cudaError_t e =
            launch_gemm_mma_list(lp, mmax <= 8 ? 1 : 2, nested8, opts ? opts->max_ctas : 0, overlap || c0 > 0, s);
        if (e != cudaSuccess) return e == cudaErrorCooperativeLaunchTooLarge ? W12_ERR_UNSUPPORTED : W12_ERR_CUDA;
    }
    return W12_OK;
}

size_t w12_tree_workspace_bytes(int32_t R, int32_t budget) {
    if (R < 1 || R > W12_TREE_MAX_REQUESTS || budget < 1 || budget > W12_TREE_MAX_BUDGET) return 0;
    return tree_workspace_bytes(R, budget);
}

w12_status w12_tree_select(const float *lp, int32_t R, int32_t D, int32_t C, int32_t budget, int32_t shared,
                           int32_t *req, int32_t *depth, uint64_t *path, float *score, int32_t *parent,
                           int32_t *count, void *workspace, size_t ws_bytes, w12_stream_t stream) {
    if (R < 1 || R > W12_TREE_MAX_REQUESTS || D < 1 || D > W12_TREE_MAX_DEPTH || C < 1 ||
        C > W12_TREE_MAX_CANDIDATES || budget < 1 || budget > W12_TREE_MAX_BUDGET || (shared != 0 && shared != 1))
        return W12_ERR_INVALID;
    if (!lp || !req || !depth || !path || !score || !parent || !count || !workspace) return W12_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(lp) & 3) || (reinterpret_cast<uintptr_t>(path) & 7) ||
        (reinterpret_cast<uintptr_t>(req) & 3) || (reinterpret_cast<uintptr_t>(depth) & 3) ||
        (reinterpret_cast<uintptr_t>(score) & 3) || (reinterpret_cast<uintptr_t>(parent) & 3) ||
        (reinterpret_cast<uintptr_t>(count) & 3) || !aligned16(workspace))
        return W12_ERR_ALIGN;
    if (ws_bytes < tree_workspace_bytes(R, budget)) return W12_ERR_CAPACITY;
    return cuda_status(launch_tree_select(lp, R, D, C, budget, shared != 0, req, depth, path, score, parent, count,
                                         workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t w12_gdn_workspace_bytes(int64_t n, int64_t H, int64_t D, int32_t mode) {
    if (n < 0 || n > W12_GDN_MAX_NODES || H < 1 || H > 65535 || (D != 64 && D != 128) ||
        (mode != W12_GDN_PATH && mode != W12_GDN_WY))
        return 0;
    return gdn_workspace_bytes(n, H, D, mode);
}

w12_status w12_gdn_tree(const float *S0, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                        const float *beta, const int32_t *parent, const int32_t *req, int64_t n, int64_t H,
                        int64_t R, int64_t D, float *o, void *workspace, size_t ws_bytes, int32_t mode,
                        w12_stream_t stream) {
    if (n < 0 || n > W12_GDN_MAX_NODES || H < 1 || H > 65535 || R < 1 || R > W12_GDN_MAX_REQUESTS ||
        (D != 64 && D != 128) || (mode != W12_GDN_PATH && mode != W12_GDN_WY))
        return W12_ERR_INVALID;
    if (!workspace || (n > 0 && (!S0 || !q || !k || !v || !alpha || !beta || !parent || !o)))
        return W12_ERR_INVALID;
    if (!aligned16(workspace) || (n > 0 && (!aligned16(S0) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
                                            !aligned16(o) || (reinterpret_cast<uintptr_t>(alpha) & 3) ||
                                            (reinterpret_cast<uintptr_t>(beta) & 3) ||
                                            (reinterpret_cast<uintptr_t>(parent) & 3) ||
                                            (reinterpret_cast<uintptr_t>(req) & 3))))
        return W12_ERR_ALIGN;
    if (ws_bytes < gdn_workspace_bytes(n, H, D, mode)) return W12_ERR_CAPACITY;
    return cuda_status(launch_gdn_tree(S0, q, k, v, alpha, beta, parent, req, (int)n, (int)H, (int)R, (int)D, o,
                                       workspace, mode, reinterpret_cast<cudaStream_t>(stream)));
}

w12_status w12_gdn_status(void *workspace, size_t ws_bytes, w12_stream_t stream) {
    if (!workspace || ws_bytes < 256) return W12_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t err = 0;
    if (cudaMemcpyAsync(&err, workspace, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    return err == 0 ? W12_OK : W12_ERR_INVALID;
}

w12_status w12_gemm_workspace_status(void *workspace, size_t ws_bytes, w12_stream_t stream) {
    if (!workspace || ws_bytes < 256) return W12_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t err = 0;
    if (cudaMemcpyAsync(&err, workspace, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    if (err == 0) return W12_OK;
    if (cudaMemsetAsync(workspace, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    return W12_ERR_TIMEOUT;
}

}  // extern "C"
