// tw_host.cu -- the fused step for tensors that live in pinned HOST memory.
//
// The token range is cut into chunks of `chunk_tokens` tokens that flow
// through two slots of a caller-provided device workspace on streams the
// library owns per device: the host->device copies of chunk i + 1 (spread over
// kH2DStreams streams, so several copy engines pull at once) overlap the
// kernel on chunk i.  When every output buffer is mapped pinned memory (the
// device can address it, which cudaHostGetDevicePointer reports), the kernel
// stores its results straight into the caller's host buffers over the host
// link, so no copy back trails the last chunk; otherwise the results are
// staged in the workspace and copied back on a third stream, overlapping the
// next chunks.  Events order the slots; the caller's stream waits for the
// last kernel or copy, so the call behaves like one asynchronous operation on
// that stream.
#include <cuda_runtime.h>

#include <mutex>

#include "tw_host.h"

namespace tw {
namespace {

constexpr size_t kAlign = 256;
constexpr int kH2DStreams = 2;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d[kH2DStreams] = {}, compute = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[2][kH2DStreams] = {}, comp_done[2] = {}, out_done[2] = {};
    std::mutex mu;  // one pipeline in flight per device at enqueue time
};

constexpr int kMaxDevices = 64;
std::mutex g_pipe_init_mu;
HostPipe g_pipes[kMaxDevices];

cudaError_t pipe_for_device(int dev, HostPipe** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    HostPipe& hp = g_pipes[dev];
    std::lock_guard<std::mutex> lock(g_pipe_init_mu);
    if (!hp.ready) {
        cudaError_t e;
        for (int i = 0; i < kH2DStreams; ++i)
            if ((e = cudaStreamCreateWithFlags(&hp.h2d[i], cudaStreamNonBlocking)) != cudaSuccess)
                return e;
        for (cudaStream_t* s : {&hp.compute, &hp.d2h})
            if ((e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t* ev : {&hp.start, &hp.end, &hp.comp_done[0], &hp.comp_done[1],
                                &hp.out_done[0], &hp.out_done[1]})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return e;
        for (int slot = 0; slot < 2; ++slot)
            for (int i = 0; i < kH2DStreams; ++i)
                if ((e = cudaEventCreateWithFlags(&hp.in_done[slot][i], cudaEventDisableTiming)) !=
                    cudaSuccess)
                    return e;
        hp.ready = true;
    }
    *out = &hp;
    return cudaSuccess;
}

}  // namespace

size_t host_workspace_bytes(int n_parts, int n_out, int64_t row_bytes, int64_t chunk_tokens) {
    const size_t chunk = round_up(static_cast<size_t>(chunk_tokens) * row_bytes);
    return round_up(static_cast<size_t>(row_bytes)) +
           2 * static_cast<size_t>(n_parts + 1 + n_out + 1) * chunk;
}

int host_pipeline(const HostCall& c, const LaunchChunk& launch_chunk, const char** what) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return *what = "cudaGetDevice", static_cast<int>(e);
    HostPipe* hp = nullptr;
    if ((e = pipe_for_device(dev, &hp)) != cudaSuccess)
        return *what = "pipeline streams", static_cast<int>(e);
    std::lock_guard<std::mutex> lock(hp->mu);

    const size_t rb = static_cast<size_t>(c.row_bytes);
    const size_t chunk = round_up(static_cast<size_t>(c.chunk_tokens) * rb);
    char* ws = static_cast<char*>(c.workspace);
    void* d_weight = ws;
    char* slot_base[2] = {ws + round_up(rb),
                          ws + round_up(rb) + static_cast<size_t>(c.n_parts + c.n_out + 2) * chunk};
    auto in_buf = [&](int slot, int r) { return slot_base[slot] + static_cast<size_t>(r) * chunk; };
    auto out_buf = [&](int slot, int k) {
        return slot_base[slot] + static_cast<size_t>(c.n_parts + 1 + k) * chunk;
    };
    const cudaStream_t user = static_cast<cudaStream_t>(c.stream);

    // Direct stores: the device address of every output host buffer.
    void* mapped_out[TW_MAX_OUTS] = {};
    void* mapped_res = nullptr;
    bool direct = cudaHostGetDevicePointer(&mapped_res, c.residual_out, 0) == cudaSuccess;
    for (int k = 0; direct && k < c.n_out; ++k)
        direct = cudaHostGetDevicePointer(&mapped_out[k], c.out[k], 0) == cudaSuccess;
    if (!direct) (void)cudaGetLastError();  // not mapped: stage and copy back

#define TW_TRY(call, name)                                     \
    do {                                                       \
        if ((e = (call)) != cudaSuccess) {                     \
            *what = name;                                      \
            return static_cast<int>(e);                        \
        }                                                      \
    } while (0)

    TW_TRY(cudaEventRecord(hp->start, user), "cudaEventRecord");
    for (int i = 0; i < kH2DStreams; ++i)
        TW_TRY(cudaStreamWaitEvent(hp->h2d[i], hp->start, 0), "cudaStreamWaitEvent");
    for (cudaStream_t s : {hp->compute, hp->d2h})
        TW_TRY(cudaStreamWaitEvent(s, hp->start, 0), "cudaStreamWaitEvent");
    TW_TRY(cudaMemcpyAsync(d_weight, c.weight, rb, cudaMemcpyHostToDevice, hp->h2d[0]),
           "cudaMemcpyAsync");

    const int64_t n_chunks = (c.t1 - c.t0 + c.chunk_tokens - 1) / c.chunk_tokens;
    for (int64_t i = 0; i < n_chunks; ++i) {
        const int slot = static_cast<int>(i & 1);
        const int64_t first = c.t0 + i * c.chunk_tokens;
        const int64_t n = c.t1 - first < c.chunk_tokens ? c.t1 - first : c.chunk_tokens;
        const size_t bytes = static_cast<size_t>(n) * rb;
        const size_t host_off = static_cast<size_t>(first) * rb;
        // The slot's previous chunk must be summed (and copied back) first.
        if (i >= 2)
            for (int j = 0; j < kH2DStreams; ++j)
                TW_TRY(cudaStreamWaitEvent(hp->h2d[j],
                                           direct ? hp->comp_done[slot] : hp->out_done[slot], 0),
                       "wait slot");
        // Input rows r = 0..n_parts (the residual last) alternate over the
        // host->device streams.
        for (int r = 0; r <= c.n_parts; ++r) {
            const void* src = r < c.n_parts ? c.partials[r] : c.residual;
            TW_TRY(cudaMemcpyAsync(in_buf(slot, r), static_cast<const char*>(src) + host_off,
                                   bytes, cudaMemcpyHostToDevice, hp->h2d[r % kH2DStreams]),
                   "cudaMemcpyAsync");
        }
        for (int j = 0; j < kH2DStreams; ++j) {
            TW_TRY(cudaEventRecord(hp->in_done[slot][j], hp->h2d[j]), "cudaEventRecord");
            TW_TRY(cudaStreamWaitEvent(hp->compute, hp->in_done[slot][j], 0),
                   "cudaStreamWaitEvent");
        }
        const void* d_parts[TW_MAX_PARTS];
        void* d_outs[TW_MAX_OUTS];
        for (int r = 0; r < c.n_parts; ++r) d_parts[r] = in_buf(slot, r);
        for (int k = 0; k < c.n_out; ++k)
            d_outs[k] = direct ? static_cast<char*>(mapped_out[k]) + host_off : out_buf(slot, k);
        void* d_res_out = direct ? static_cast<char*>(mapped_res) + host_off
                                 : static_cast<void*>(out_buf(slot, c.n_out));
        const int rc = launch_chunk(d_parts, in_buf(slot, c.n_parts), d_weight, d_outs,
                                    d_res_out, n, hp->compute);
        if (rc != 0) return *what = nullptr, rc;  // a tw_status, message already set
        TW_TRY(cudaEventRecord(hp->comp_done[slot], hp->compute), "cudaEventRecord");
        if (direct) continue;

        TW_TRY(cudaStreamWaitEvent(hp->d2h, hp->comp_done[slot], 0), "cudaStreamWaitEvent");
        for (int k = 0; k < c.n_out; ++k)
            TW_TRY(cudaMemcpyAsync(static_cast<char*>(c.out[k]) + host_off, out_buf(slot, k),
                                   bytes, cudaMemcpyDeviceToHost, hp->d2h),
                   "cudaMemcpyAsync");
        TW_TRY(cudaMemcpyAsync(static_cast<char*>(c.residual_out) + host_off,
                               out_buf(slot, c.n_out), bytes, cudaMemcpyDeviceToHost, hp->d2h),
               "cudaMemcpyAsync");
        TW_TRY(cudaEventRecord(hp->out_done[slot], hp->d2h), "cudaEventRecord");
    }
    // The caller's stream continues after the last kernel (direct stores) or
    // the last copy back; the copies in and the kernels precede it through
    // the events.
    TW_TRY(cudaEventRecord(hp->end, direct ? hp->compute : hp->d2h), "cudaEventRecord");
    TW_TRY(cudaStreamWaitEvent(user, hp->end, 0), "cudaStreamWaitEvent");
#undef TW_TRY
    return 0;
}

}  // namespace tw
