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

#include <cstdio>
#include <mutex>
#include <string>

#include "tw.h"
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

}  // namespace

extern "C" int tw_fused_reduce_add_rmsnorm_host_noalloc(
    const void* const* partials, int n_parts, const void* residual, const void* weight,
    void* const* out, int n_out, void* residual_out, int64_t T, int64_t H, float eps,
    int64_t t0, int64_t t1, int max_sms, int64_t chunk_tokens, void* stream, int dtype) {
    // Pick the largest chunk that fits the array when none is given.
    if (chunk_tokens <= 0) {
        size_t one = 0;
        int rc = tw_host_workspace_bytes(n_parts, n_out, H, 1, dtype, &one);
        if (rc != TW_OK) return rc;
        size_t two = 0;
        rc = tw_host_workspace_bytes(n_parts, n_out, H, 2, dtype, &two);
        if (rc != TW_OK) return rc;
        const size_t per_token = two - one;  // bytes the workspace grows per chunk token
        if (one > kNoAllocScratchBytes) chunk_tokens = 1;  // refused just below
        else chunk_tokens = static_cast<int64_t>(1 + (kNoAllocScratchBytes - one) / per_token);
    }
    size_t need = 0;
    int rc = tw_host_workspace_bytes(n_parts, n_out, H, chunk_tokens, dtype, &need);
    if (rc != TW_OK) return rc;
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
