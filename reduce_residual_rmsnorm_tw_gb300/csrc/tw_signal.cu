// tw_signal.cu -- the producer side of the readiness flags: raise a range of
// token-block flags to an epoch with release semantics (the FLUX notes'
// SetSignal, paired with the WaitSignal of tw_fused_reduce_add_rmsnorm_flags).
//
// Work queued earlier on the stream (the kernels or copies that wrote the
// blocks' partial and residual rows) has completed before this kernel starts;
// each flag is then written with st.release at GPU scope, so a consumer that
// reads the flag with an acquire load at GPU scope also sees those rows.  A
// plain store or memset of the flag gives no such guarantee: it is a weak
// store, not a release.
#include <cuda_runtime.h>

#include <cstdio>

#include "tw.h"
#include "tw_internal.h"

namespace tw {
namespace {

constexpr int kSignalThreads = 256;
constexpr int kSignalMaxBlocks = 64;

__global__ void __launch_bounds__(kSignalThreads)
    set_ready_kernel(unsigned int* ready, int64_t n, unsigned int epoch) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ready + i), "r"(epoch)
                     : "memory");
}

}  // namespace

int signal_prepare() {
    // Loads the kernel now: with lazy module loading a kernel is loaded at its
    // first launch, and that load may wait for kernels already running -- a
    // consumer spinning on the very flags this kernel would raise.
    cudaFuncAttributes attr;
    return static_cast<int>(cudaFuncGetAttributes(&attr, set_ready_kernel));
}

}  // namespace tw

extern "C" int tw_set_ready(uint32_t* ready, int64_t first_block, int64_t n_blocks,
                            uint32_t epoch, void* stream) {
    if (!ready) return tw::set_last_error(TW_ERR_INVALID_ARG, "ready is NULL");
    if ((reinterpret_cast<uintptr_t>(ready) & 3u) != 0)
        return tw::set_last_error(TW_ERR_ALIGNMENT, "ready must be 4-byte aligned");
    if (first_block < 0 || n_blocks < 0 || first_block > (int64_t{1} << 46) ||
        n_blocks > (int64_t{1} << 46))
        return tw::set_last_error(TW_ERR_INVALID_ARG,
                                  "first_block and n_blocks must be in [0, 2^46]");
    if (n_blocks == 0) return TW_OK;
    int64_t blocks = (n_blocks + tw::kSignalThreads - 1) / tw::kSignalThreads;
    if (blocks > tw::kSignalMaxBlocks) blocks = tw::kSignalMaxBlocks;
    tw::set_ready_kernel<<<static_cast<unsigned>(blocks), tw::kSignalThreads, 0,
                           static_cast<cudaStream_t>(stream)>>>(ready + first_block, n_blocks,
                                                                epoch);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char buf[160];
        snprintf(buf, sizeof(buf), "set_ready launch: %s (%s)", cudaGetErrorName(e),
                 cudaGetErrorString(e));
        return tw::set_last_error(TW_ERR_CUDA, buf);
    }
    return TW_OK;
}
