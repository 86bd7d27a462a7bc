// tw_noalloc.cu -- the host-buffer fused step for callers that cannot
// allocate device memory.
//
// tw_fused_reduce_add_rmsnorm_host needs a device workspace from its caller.
// Some callers cannot provide one: a host program that talks to the GPU only
// through this library's C ABI and has no CUDA allocator of its own, a
// process whose device memory is reserved up front by a framework that does
// not hand out raw buffers, or code running where cudaMalloc is not allowed
// (for instance inside a stream capture, or under a policy that forbids
// device allocation after start-up).  This entry point takes its staging
// workspace from one file-scope device array instead, so it allocates
// nothing.  The array exists once per GPU that loads the library and lives
// until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "tw.h"
#include "tw_host.h"
#include "tw_internal.h"

namespace {

// Maximum staging workspace of the no-allocation entry point (per GPU).
constexpr size_t kNoAllocScratchBytes = TW_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the array's name is only a host-side stand-in).
int scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return static_cast<int>(e);
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return 0;
}

// Staging bytes for chunks of k tokens, or SIZE_MAX if the query refuses k.
size_t staging_bytes(int n_parts, int n_out, int64_t H, int dtype, int64_t k) {
    size_t need = 0;
    return tw_host_workspace_bytes(n_parts, n_out, H, k, dtype, &need) == TW_OK ? need : SIZE_MAX;
}

// The largest chunk in [1, span] whose staging fits the array, or 0 if not
// even one token's does.  The staging size grows with the chunk (each chunk
// buffer is rounded up to 256 bytes, so not by a fixed amount per token):
// bisection over that monotone size, not an estimate of its slope.
int64_t largest_fitting_chunk(int n_parts, int n_out, int64_t H, int dtype, int64_t span) {
    if (staging_bytes(n_parts, n_out, H, dtype, 1) > kNoAllocScratchBytes) return 0;
    int64_t lo = 1, hi = span;  // chunks of lo tokens fit
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo + 1) / 2;
        if (staging_bytes(n_parts, n_out, H, dtype, mid) <= kNoAllocScratchBytes) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

}  // namespace

extern "C" int tw_fused_reduce_add_rmsnorm_host_noalloc(
    const void* const* partials, int n_parts, const void* residual, const void* weight,
    void* const* out, int n_out, void* residual_out, int64_t T, int64_t H, float eps,
    int64_t t0, int64_t t1, int max_sms, int64_t chunk_tokens, void* stream, int dtype) {
    int rc = tw::check_host_args(partials, n_parts, residual, weight, out, n_out, residual_out,
                                 T, H, eps, t0, t1, max_sms, dtype);
    if (rc != TW_OK) return rc;
    if (t0 == t1) return TW_OK;
    // A chunk never needs to be longer than the range.
    const int64_t span = t1 - t0;
    if (chunk_tokens <= 0) {
        // The largest chunk that fits the array.
        chunk_tokens = largest_fitting_chunk(n_parts, n_out, H, dtype, span);
        if (chunk_tokens == 0) chunk_tokens = 1;  // refused just below
    } else if (chunk_tokens > span) {
        chunk_tokens = span;
    }
    const size_t need = staging_bytes(n_parts, n_out, H, dtype, chunk_tokens);
    if (need > kNoAllocScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof(buf),
                 "the no-allocation entry point needs %zu bytes of staging for chunks of %lld "
                 "tokens; its device array holds %zu bytes (use smaller chunks)",
                 need, (long long)chunk_tokens, kNoAllocScratchBytes);
        return tw::set_last_error(TW_ERR_UNSUPPORTED, buf);
    }
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != 0) {
        const std::string msg = std::string("cudaGetSymbolAddress: ") +
                                cudaGetErrorName(static_cast<cudaError_t>(rc));
        return tw::set_last_error(TW_ERR_CUDA, msg.c_str());
    }
    return tw_fused_reduce_add_rmsnorm_host(partials, n_parts, residual, weight, out, n_out,
                                            residual_out, T, H, eps, t0, t1, max_sms, scratch,
                                            kNoAllocScratchBytes, chunk_tokens, stream, dtype);
}
