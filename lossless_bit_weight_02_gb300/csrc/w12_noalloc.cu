// w12_gemm_noalloc: the W12 GEMM for callers that cannot allocate device
// memory.
//
// Some hosts of this library own every byte of device memory themselves: an
// inference engine that plans its memory once at start-up and forbids any
// allocation afterwards, a plug-in running inside another framework's memory
// pool, or a latency-critical loop where cudaMalloc's implicit device
// synchronisation would stall work on other streams.  Such callers cannot
// provide the split-K workspace that w12_gemm asks for.  This entry point
// uses a scratch buffer that lives in the library itself instead: a
// file-scope device array of W12_NOALLOC_SCRATCH_BYTES, which every GPU that
// loads the library holds until the process exits.
//
// The host-side name of the array is only a stand-in for it; its device
// address comes from cudaGetSymbolAddress, asked on every call for the
// device current at the time (so a reset or recreated context never leaves a
// stale address behind).  The very first lookup on a device loads the
// library's device code there, which is why the first call on a device
// should come before any stream capture.
#include <cstdint>

#include <cuda_runtime.h>

#include "w12.h"
#include "w12_internal.h"

namespace {

constexpr size_t kScratchBytes = W12_NOALLOC_SCRATCH_BYTES;
// Bytes at the front of a w12_gemm workspace that must be zero when a call
// starts: the error word and the split-K arrival counters.
constexpr size_t kZeroedPrefix = w12::kWsPartialsOff;
static_assert(kZeroedPrefix < kScratchBytes, "the scratch must hold the zeroed prefix");

static __device__ __align__(256) unsigned char g_w12_scratch[kScratchBytes];

// Device address of the scratch array on the current device.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_w12_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" w12_status w12_gemm_noalloc(const uint16_t *A, int64_t lda, const w12_tensor *w, uint16_t *Y,
                                       int64_t ldy, int64_t M, const w12_gemm_opts *opts,
                                       w12_stream_t stream) {
    if (!w || M < 0 || w->N < 0 || w->K < 0) return W12_ERR_INVALID;
    if (M == 0 || w->N == 0) return W12_OK;
    size_t need = 0;
    const w12_status st = w12::gemm_plan_bytes(M, w->N, w->K, opts, &need);
    if (st != W12_OK) return st;                        // what w12_gemm returns for these options
    if (need > kScratchBytes) return W12_ERR_CAPACITY;  // beyond the built-in scratch
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return W12_ERR_CUDA;
    // The previous call may have failed part-way; start from clean counters
    // and a clear error word.
    const size_t zero = need < kZeroedPrefix ? need : kZeroedPrefix;
    if (cudaMemsetAsync(scratch, 0, zero, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W12_ERR_CUDA;
    return w12_gemm(A, lda, w, Y, ldy, M, scratch, kScratchBytes, opts, stream);
}

extern "C" w12_status w12_gemm_noalloc_status(w12_stream_t stream) {
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return W12_ERR_CUDA;
    return w12_gemm_workspace_status(scratch, kScratchBytes, stream);
}
