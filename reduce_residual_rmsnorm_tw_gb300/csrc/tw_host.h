// tw_host.h -- host-memory pipeline shared between tw_host.cu and the API.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>

#include "tw.h"

namespace tw {

// One host-buffer call: HOST pointers for the tensors, a DEVICE workspace.
struct HostCall {
    const void* const* partials;
    int n_parts;
    const void* residual;
    const void* weight;
    void* const* out;
    int n_out;
    void* residual_out;
    int64_t row_bytes;
    int64_t t0, t1;
    int64_t chunk_tokens;
    void* workspace;
    void* stream;
};

// Launch the fused kernel on one staged chunk of n tokens (device pointers,
// rows [0, n)) on `stream`; returns a tw_status.
using LaunchChunk = std::function<int(const void* const* partials, const void* residual,
                                      const void* weight, void* const* out, void* residual_out,
                                      int64_t n, cudaStream_t stream)>;

// Bytes of device workspace the pipeline needs.
size_t host_workspace_bytes(int n_parts, int n_out, int64_t row_bytes, int64_t chunk_tokens);

// The argument rules of tw.h for one call (no CUDA call): TW_OK, or the
// status with the calling thread's error message set.
int check_host_args(const void* const* partials, int n_parts, const void* residual,
                    const void* weight, void* const* out, int n_out, void* residual_out,
                    int64_t T, int64_t H, float eps, int64_t t0, int64_t t1, int max_sms,
                    int dtype);

// Enqueue the pipeline.  Returns 0, a cudaError_t value with *what naming the
// failing call, or a tw_status from launch_chunk with *what == nullptr.
int host_pipeline(const HostCall& c, const LaunchChunk& launch_chunk, const char** what);

}  // namespace tw
