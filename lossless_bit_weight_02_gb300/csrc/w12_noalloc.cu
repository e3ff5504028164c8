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
// address comes from cudaGetSymbolAddress, called once per device (with that
// device current) on the first call of this entry point on that device.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "w12.h"

namespace {

constexpr size_t kScratchBytes = W12_NOALLOC_SCRATCH_BYTES;
// Bytes at the front of a w12_gemm workspace that must be zero when a call
// starts: the error word (256 bytes) and the split-K arrival counters
// (4 bytes for each of at most 65536 row stripes).
constexpr size_t kZeroedPrefix = 256 + 4 * 65536;

static __device__ __align__(256) unsigned char g_w12_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_w12_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" w12_status w12_gemm_noalloc(const uint16_t *A, int64_t lda, const w12_tensor *w, uint16_t *Y,
                                       int64_t ldy, int64_t M, const w12_gemm_opts *opts,
                                       w12_stream_t stream) {
    if (!w || M < 0 || w->N < 0 || w->K < 0) return W12_ERR_INVALID;
    if (M == 0 || w->N == 0) return W12_OK;
    const size_t need = w12_gemm_workspace_bytes(M, w->N, w->K, opts);
    if (need == 0) return W12_ERR_INVALID;          // the shape or the options are not supported
    if (need > kScratchBytes) return W12_ERR_CAPACITY;  // beyond the built-in scratch
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return W12_ERR_CUDA;
    // The previous call may have failed part-way; start from clean counters.
    const size_t zero = need < kZeroedPrefix ? need : kZeroedPrefix;
    if (cudaMemsetAsync(scratch, 0, zero, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W12_ERR_CUDA;
    return w12_gemm(A, lda, w, Y, ldy, M, scratch, kScratchBytes, opts, stream);
}
