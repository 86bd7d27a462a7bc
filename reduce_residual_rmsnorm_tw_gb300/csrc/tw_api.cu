// tw_api.cu -- the C ABI of libtw.so: argument checks, per-device state,
// kernel choice and the two-stream token split.  Every rule stated in tw.h is
// checked here on the host before the first CUDA call of an entry point.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "tw.h"
#include "tw_host.h"
#include "tw_internal.h"

namespace tw {
namespace {

// Bounded-wait give-ups of any kernel on this device (see tw_device_status).
__device__ unsigned int g_status_word;
// Work counter pairs of the rows kernel (next unit, CTAs done); each launch
// that claims units leaves its pair at zero when it ends.
__device__ unsigned int g_work[2 * kWorkSlots];

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TW_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Under TW_PATH_AUTO, a token range goes to the cluster kernel (one cluster
// per token) when every one of its clusters can run at once -- at most
// DeviceState::max_clusters clusters of the launch's size and kernel
// instantiation, the count from the occupancy API (a cluster must fit in one
// GPC; on a GB300 with 152 SMs twelve 8-CTA clusters took 3.1 us, sixteen 5.6
// us, the rows kernel 4.2 us) -- and to the rows kernel otherwise.  kClusterPathMaxTokens is the
// bound used if the device cannot be asked.  The warp kernel is never faster
// on this GPU (one warp cannot pull a 100+ KB token quickly) and runs only
// when asked for.
constexpr int64_t kClusterPathMaxTokens = 8;
// AUTO never takes the cluster kernel beyond this many tokens (measured on
// N = 8, H = 8192 bf16: at 128 tokens it still beat the rows kernel, 5.65
// vs 5.8 us; at 152 it lost, 8.1 vs 6.6 us).
constexpr int64_t kClusterAutoMaxTokens = 128;
// Rows launches claim units from a work counter when they have at least this
// many CTAs and units per CTA (on a GB300 this took the 8192- and 16384-token
// workloads 5-10 % faster; launches of ~7 units per CTA or on a few SMs gained
// nothing and lost to the counter's bookkeeping).
constexpr int64_t kClaimMinGrid = 64;
constexpr int64_t kClaimMinUnits = 16;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;
    bool cluster_ready = false;
    const char* cluster_error = "";
    // Clusters of 1, 2, 4, 8 CTAs that run at once, per kernel instantiation:
    // [0] with every CTA alone on its SM (budgeted launches), [1] with CTAs
    // free to share SMs; then [log2 cluster][dtype][vectors per thread 1, 2,
    // 4][partials held 2, 4, 8, 16].
    int max_clusters[2][4][2][3][4] = {};
    unsigned int* status = nullptr;
    cudaEvent_t fork = nullptr;
    cudaEvent_t join = nullptr;
    std::mutex split_mu;  // orders the record/wait pairs of concurrent splits
    // Work counter pairs: the device array, and per pair the event recorded
    // after the last launch that used it (a pair is handed out again only
    // once its event has completed).
    unsigned int* work = nullptr;
    cudaEvent_t work_done[kWorkSlots] = {};
    bool work_used[kWorkSlots] = {};
    bool work_bad[kWorkSlots] = {};
    int work_next = 0;
    std::mutex work_mu;
};

constexpr int kMaxDevices = 64;
std::mutex g_init_mu;
DeviceState g_devices[kMaxDevices];

int device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(TW_ERR_UNSUPPORTED, "device %d", dev);
    DeviceState& d = g_devices[dev];
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (!d.ready) {
        int major = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major < 10)
            return fail(TW_ERR_UNSUPPORTED, "device %d has compute capability %d.x; "
                        "libtw.so is built for sm_103a", dev, major);
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (d.smem_optin < kExclusiveSmemBytes)
            return fail(TW_ERR_UNSUPPORTED, "device %d allows only %d bytes of shared memory",
                        dev, d.smem_optin);
        if ((e = static_cast<cudaError_t>(rows_set_smem_limit(d.smem_optin))) != cudaSuccess ||
            (e = static_cast<cudaError_t>(warp_set_smem_limit(d.smem_optin))) != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute");
        // Every kernel of the library is loaded here, before any of them can
        // be waiting for another (lazy loading would load tw_set_ready's at
        // its first launch, which may wait for running kernels).
        if ((e = static_cast<cudaError_t>(signal_prepare())) != cudaSuccess)
            return cuda_fail(e, "cudaFuncGetAttributes");
        // The cluster kernel is optional: if it cannot be configured, that
        // path reports TW_ERR_UNSUPPORTED and the others still run.
        e = static_cast<cudaError_t>(cluster_set_attributes(d.smem_optin));
        d.cluster_ready = e == cudaSuccess;
        if (e != cudaSuccess) {
            d.cluster_error = cudaGetErrorName(e);
            (void)cudaGetLastError();  // clear the (non-sticky) launch-API error
        }
        for (int shared = 0; shared < 2; ++shared)
            for (int i = 0; d.cluster_ready && i < 4; ++i)
                for (int dt = 0; dt < 2; ++dt)
                    for (int v = 0; v < 3; ++v)
                        for (int q = 0; q < 4; ++q) {
                            int n = 0;
                            if (cluster_max_active(1 << i, shared ? 0 : kExclusiveSmemBytes, dt,
                                                   1 << v, 2 << q, &n) != cudaSuccess ||
                                n < 1) {
                                (void)cudaGetLastError();
                                n = static_cast<int>(kClusterPathMaxTokens);
                            }
                            d.max_clusters[shared][i][dt][v][q] = n;
                        }
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress");
        if ((e = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "cudaEventCreateWithFlags");
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.work), g_work)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress");
        for (int k = 0; k < kWorkSlots; ++k)
            if ((e = cudaEventCreateWithFlags(&d.work_done[k], cudaEventDisableTiming)) !=
                cudaSuccess)
                return cuda_fail(e, "cudaEventCreateWithFlags");
        d.ready = true;
    }
    *out = &d;
    return TW_OK;
}

struct Args {
    const void* const* partials;
    int n_parts;
    const void* residual;
    const void* weight;
    void* const* out;
    int n_out;
    void* residual_out;
    int64_t T, H;
    float eps;
    int64_t t0, t1;
    int max_sms;
    int dtype;
    int colsplit = 0;
    int host_direct = 0;  // tensors in mapped host memory, read in place
    const unsigned int* ready = nullptr;  // readiness flags (rows kernel only)
    int64_t block_tokens = 0;
    unsigned int epoch = 0;
};

size_t elem_size(int dtype) { return dtype == TW_BF16 ? 2 : 4; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na != 0 && nb != 0 && a0 < b0 + nb && b0 < a0 + na;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// All host-side rules of tw.h; no CUDA call.
int check_args(const Args& a) {
    if (a.dtype != TW_BF16 && a.dtype != TW_F32)
        return fail(TW_ERR_INVALID_ARG, "dtype %d is not TW_BF16 or TW_F32", a.dtype);
    if (!a.partials || !a.out || !a.residual || !a.weight || !a.residual_out)
        return fail(TW_ERR_INVALID_ARG, "NULL pointer argument");
    if (a.n_parts < 1 || a.n_parts > TW_MAX_PARTS)
        return fail(TW_ERR_INVALID_ARG, "n_parts %d outside [1, %d]", a.n_parts, TW_MAX_PARTS);
    if (a.n_out < 1 || a.n_out > TW_MAX_OUTS)
        return fail(TW_ERR_INVALID_ARG, "n_out %d outside [1, %d]", a.n_out, TW_MAX_OUTS);
    for (int r = 0; r < a.n_parts; ++r)
        if (!a.partials[r]) return fail(TW_ERR_INVALID_ARG, "partials[%d] is NULL", r);
    for (int k = 0; k < a.n_out; ++k)
        if (!a.out[k]) return fail(TW_ERR_INVALID_ARG, "out[%d] is NULL", k);
    const int64_t max_h = a.dtype == TW_BF16 ? TW_MAX_H_BF16 : TW_MAX_H_F32;
    if (a.T < 0 || a.H < 1)
        return fail(TW_ERR_INVALID_ARG, "T %lld and H %lld must satisfy T >= 0, H >= 1",
                    (long long)a.T, (long long)a.H);
    if (a.H > max_h)
        return fail(TW_ERR_UNSUPPORTED, "H %lld above the limit %lld for this dtype",
                    (long long)a.H, (long long)max_h);
    // A buffer's byte span must be a plausible device address range, so that
    // T * H * size and every pointer + offset below stay far from overflow.
    if (a.T > (int64_t{1} << 48) / (a.H * static_cast<int64_t>(elem_size(a.dtype))))
        return fail(TW_ERR_INVALID_ARG, "T %lld x H %lld buffers exceed 2^48 bytes",
                    (long long)a.T, (long long)a.H);
    if (a.t0 < 0 || a.t0 > a.t1 || a.t1 > a.T)
        return fail(TW_ERR_INVALID_ARG, "token range [%lld, %lld) not within [0, %lld]",
                    (long long)a.t0, (long long)a.t1, (long long)a.T);
    if (!(a.eps >= 0.f) || std::isinf(a.eps))
        return fail(TW_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (a.max_sms < 1) return fail(TW_ERR_INVALID_ARG, "max_sms %d < 1", a.max_sms);

    const size_t es = elem_size(a.dtype);
    if ((static_cast<size_t>(a.H) * es) % 16 != 0)
        return fail(TW_ERR_ALIGNMENT, "H * element size (%lld bytes) is not a multiple of 16",
                    (long long)(a.H * static_cast<int64_t>(es)));
    if (misaligned(a.residual) || misaligned(a.weight) || misaligned(a.residual_out))
        return fail(TW_ERR_ALIGNMENT, "residual, weight and residual_out must be 16-byte aligned");
    for (int r = 0; r < a.n_parts; ++r)
        if (misaligned(a.partials[r]))
            return fail(TW_ERR_ALIGNMENT, "partials[%d] is not 16-byte aligned", r);
    for (int k = 0; k < a.n_out; ++k)
        if (misaligned(a.out[k])) return fail(TW_ERR_ALIGNMENT, "out[%d] is not 16-byte aligned", k);

    if (a.colsplit) {
        // Each rank's column slice must start and end on a 16-byte boundary.
        for (int r = 0; r <= a.n_parts; ++r)
            if (((a.H * r / a.n_parts) * static_cast<int64_t>(es)) % 16 != 0)
                return fail(TW_ERR_ALIGNMENT, "column slice %d of H %lld over %d ranks does not "
                            "start on a 16-byte boundary", r, (long long)a.H, a.n_parts);
    }

    // Aliasing: outputs against inputs and against each other.
    const size_t tb = static_cast<size_t>(a.T) * static_cast<size_t>(a.H) * es;
    const size_t wb = static_cast<size_t>(a.H) * es;
    const int n_outputs = a.n_out + 1;
    for (int i = 0; i < n_outputs; ++i) {
        const void* o = i < a.n_out ? a.out[i] : a.residual_out;
        const bool is_res_out = i == a.n_out;
        for (int r = 0; r < a.n_parts; ++r)
            if (overlaps(o, tb, a.partials[r], tb))
                return fail(TW_ERR_ALIAS, "an output overlaps partials[%d]", r);
        if (overlaps(o, tb, a.weight, wb)) return fail(TW_ERR_ALIAS, "an output overlaps weight");
        if (overlaps(o, tb, a.residual, tb) && !(is_res_out && o == a.residual))
            return fail(TW_ERR_ALIAS, "an output overlaps residual (only residual_out == "
                        "residual, exactly, is allowed)");
        for (int j = i + 1; j < n_outputs; ++j) {
            const void* o2 = j < a.n_out ? a.out[j] : a.residual_out;
            if (overlaps(o, tb, o2, tb)) return fail(TW_ERR_ALIAS, "two outputs overlap");
        }
    }
    return TW_OK;
}

Params make_params(const Args& a, const DeviceState& d, int64_t t0, int64_t t1,
                   uint32_t* smid_log) {
    Params p{};
    for (int r = 0; r < a.n_parts; ++r) p.partials[r] = a.partials[r];
    for (int k = 0; k < a.n_out; ++k) p.out[k] = a.out[k];
    p.residual = a.residual;
    p.weight = a.weight;
    p.residual_out = a.residual_out;
    p.smid_log = smid_log;
    p.status = d.status;
    p.t0 = t0;
    p.t1 = t1;
    p.H = a.H;
    p.row_bytes = a.H * static_cast<int64_t>(elem_size(a.dtype));
    p.n_parts = a.n_parts;
    p.n_out = a.n_out;
    p.colsplit = a.colsplit;
    p.ready = a.ready;
    p.block_tokens = a.block_tokens;
    p.epoch = a.epoch;
    const int64_t es = static_cast<int64_t>(elem_size(a.dtype));
    for (int r = 0; r <= a.n_parts; ++r) p.col_lo[r] = (a.H * r / a.n_parts) * es;
    p.eps = a.eps;
    p.inv_H = static_cast<float>(1.0 / static_cast<double>(a.H));
    return p;
}

// A work counter pair for a rows launch on `stream`, or -1 for a fixed
// schedule: while the stream is being captured into a CUDA graph (a graph
// replays the same pair, and no event can be polled), or when every pair is
// still in use by a launch that has not completed.  Called with work_mu held.
int acquire_work_slot(DeviceState& d, void* stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (cs != cudaStreamCaptureStatusNone) return -1;
    for (int n = 0; n < kWorkSlots; ++n) {
        const int k = (d.work_next + n) % kWorkSlots;
        if (d.work_bad[k]) continue;
        if (d.work_used[k]) {
            const cudaError_t e = cudaEventQuery(d.work_done[k]);
            if (e == cudaErrorNotReady) continue;
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                continue;
            }
        }
        d.work_next = (k + 1) % kWorkSlots;
        return k;
    }
    return -1;
}

// Launch one kernel over rows [t0, t1) (non-empty) on `stream`.
int launch_range(const Args& a, DeviceState& d, int64_t t0, int64_t t1, int path,
                 uint32_t* smid_log, void* stream) {
    const int64_t tokens = t1 - t0;
    const int64_t sms = a.max_sms < d.sm_count ? a.max_sms : d.sm_count;
    // A launch that may use every SM overlaps its start with the previous
    // kernel's drain; a budgeted launch does not, so that at no time more than
    // max_sms SMs hold its CTAs.
    const bool pdl = a.max_sms >= d.sm_count;
    Params p = make_params(a, d, t0, t1, smid_log);
    // L2 warming is for device memory; host-resident rows are read once,
    // in place.
    p.prefetch = pdl && !a.host_direct ? 1 : 0;
    // Largest power-of-two cluster within the budget (at most 8: portable).
    int cluster = 1;
    while (cluster * 2 <= 8 && cluster * 2 <= sms) cluster *= 2;
    const bool cluster_ok =
        d.cluster_ready && cluster_vectors_per_thread(p.row_bytes, cluster) != 0;
    if (a.colsplit || a.ready) {
        if (path != TW_PATH_AUTO && path != TW_PATH_ROWS)
            return fail(TW_ERR_UNSUPPORTED,
                        "the column-split mode and readiness flags run on the rows kernel only");
        path = TW_PATH_ROWS;
    }
    // Host-resident tensors are read with plain loads (the cluster kernel):
    // the rows kernel's bulk copies are kept to device memory.
    if (a.host_direct) path = TW_PATH_CLUSTER;
    int log2c = 0;
    while ((2 << log2c) <= cluster) ++log2c;
    // Clusters of this launch's instantiation that run at once with every CTA
    // alone on its SM, and (launches without a budget only) with CTAs
    // sharing SMs.
    int64_t alone = 0, shared = 0;
    if (cluster_ok) {
        int v = 0, q = 0;
        while ((2 << v) <= cluster_vectors_per_thread(p.row_bytes, cluster)) ++v;
        while ((4 << q) <= cluster_np(p.n_parts)) ++q;
        const int dt = a.dtype == TW_BF16 ? 0 : 1;
        alone = d.max_clusters[0][log2c][dt][v][q];
        shared = pdl ? d.max_clusters[1][log2c][dt][v][q] : 0;
    }
    if (path == TW_PATH_AUTO) {
        const bool fits = pdl ? tokens <= (alone > shared ? alone : shared)
                              : tokens <= alone && tokens * cluster <= sms;
        path = (tokens <= kClusterAutoMaxTokens && fits && cluster_ok) ? TW_PATH_CLUSTER
                                                                       : TW_PATH_ROWS;
    }

    int err;
    if (path == TW_PATH_ROWS) {
        p.unit_tokens = rows_unit_tokens(p, tokens, sms);
        const size_t smem = rows_plan(p, d.smem_optin);
        if (smem == 0)
            return fail(TW_ERR_UNSUPPORTED, "shared memory too small for rows of %lld bytes",
                        (long long)p.row_bytes);
        const int64_t units = (tokens + p.unit_tokens - 1) / p.unit_tokens;
        const int grid = static_cast<int>(units < sms ? units : sms);
        // Claimed units (a work counter pair of its own) for long launches on
        // many SMs, where CTAs streaming at different speeds would otherwise
        // finish far apart: at least kClaimMinGrid CTAs and kClaimMinUnits
        // units per CTA (and fewer than 2^31 units, the counter's range).
        // Shorter launches cannot rebalance by whole units and pay the
        // counter's host-side bookkeeping; readiness flags keep the fixed
        // schedule.
        if (a.ready || grid < kClaimMinGrid || units < kClaimMinUnits * grid ||
            units >= (int64_t{1} << 31)) {
            p.pipes = rows_two_pipes_fit(p, a.max_sms < d.sm_count) ? 2 : 1;
            err = launch_rows(p, a.dtype, grid, smem, pdl, stream);
        } else {
            std::lock_guard<std::mutex> lock(d.work_mu);
            const int slot = acquire_work_slot(d, stream);
            p.work = slot >= 0 ? d.work + 2 * slot : nullptr;
            err = launch_rows(p, a.dtype, grid, smem, pdl, stream);
            if (slot >= 0 && err == cudaSuccess) {
                if (cudaEventRecord(d.work_done[slot], static_cast<cudaStream_t>(stream)) !=
                    cudaSuccess) {
                    // Without its event the pair could be handed out while
                    // this launch runs: never use it again.
                    (void)cudaGetLastError();
                    d.work_bad[slot] = true;
                } else {
                    d.work_used[slot] = true;
                }
            }
        }
    } else if (path == TW_PATH_WARP) {
        const int64_t ctas = (tokens + kWarpTokensPerCta - 1) / kWarpTokensPerCta;
        const int grid = static_cast<int>(ctas < sms ? ctas : sms);
        const size_t xs = warp_stage_bytes(p.row_bytes, a.dtype);
        const bool staged = xs <= static_cast<size_t>(d.smem_optin);
        const size_t smem =
            staged && xs > static_cast<size_t>(kExclusiveSmemBytes) ? xs : kExclusiveSmemBytes;
        err = launch_warp(p, a.dtype, grid, smem, staged, pdl, stream);
    } else if (path == TW_PATH_CLUSTER) {
        if (!d.cluster_ready)
            return fail(TW_ERR_UNSUPPORTED, "cluster kernel unavailable on this device (%s)",
                        d.cluster_error);
        if (!cluster_ok)
            return fail(TW_ERR_UNSUPPORTED, "row of %lld bytes too long for a cluster of %d",
                        (long long)p.row_bytes, cluster);
        // One CTA per SM (the exclusive shared-memory request) under a budget
        // and whenever the clusters fit that way; otherwise, without a
        // budget, CTAs share SMs so that more clusters run at once.
        const bool share = pdl && tokens > alone && shared > sms / cluster;
        int64_t max_clusters = share ? shared : sms / cluster;
        const int n_clusters = static_cast<int>(tokens < max_clusters ? tokens : max_clusters);
        err = launch_cluster(p, a.dtype, cluster, n_clusters, share ? 0 : kExclusiveSmemBytes,
                             pdl, stream);
    } else {
        return fail(TW_ERR_INVALID_ARG, "unknown path %d", path);
    }
    if (err != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(err), "kernel launch");
    return TW_OK;
}

int fused(const Args& a, int path, uint32_t* smid_log, void* stream) {
    int rc = check_args(a);
    if (rc != TW_OK) return rc;
    if (path < TW_PATH_AUTO || path > TW_PATH_CLUSTER)
        return fail(TW_ERR_INVALID_ARG, "unknown path %d", path);
    if (a.t0 == a.t1) return TW_OK;
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != TW_OK) return rc;
    return launch_range(a, *d, a.t0, a.t1, path, smid_log, stream);
}

bool is_pinned_host(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeHost;
}

// chunk_tokens == 0: one launch whose kernel reads the host tensors in place
// and stores straight into the host outputs, through their device mappings.
int fused_in_place_from_host(const Args& a, void* stream) {
    if (a.t0 == a.t1) return TW_OK;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != TW_OK) return rc;
    const void* m_parts[TW_MAX_PARTS];
    void* m_out[TW_MAX_OUTS];
    void* m_res = nullptr;
    void* m_weight = nullptr;
    void* m_res_out = nullptr;
    bool mapped = true;
    for (int r = 0; mapped && r < a.n_parts; ++r) {
        void* m = nullptr;
        mapped = is_pinned_host(a.partials[r]) &&
                 cudaHostGetDevicePointer(&m, const_cast<void*>(a.partials[r]), 0) == cudaSuccess;
        m_parts[r] = m;
    }
    for (int k = 0; mapped && k < a.n_out; ++k)
        mapped = is_pinned_host(a.out[k]) &&
                 cudaHostGetDevicePointer(&m_out[k], a.out[k], 0) == cudaSuccess;
    mapped = mapped && is_pinned_host(a.residual) && is_pinned_host(a.weight) &&
             is_pinned_host(a.residual_out) &&
             cudaHostGetDevicePointer(&m_res, const_cast<void*>(a.residual), 0) == cudaSuccess &&
             cudaHostGetDevicePointer(&m_weight, const_cast<void*>(a.weight), 0) == cudaSuccess &&
             cudaHostGetDevicePointer(&m_res_out, a.residual_out, 0) == cudaSuccess;
    if (!mapped) {
        (void)cudaGetLastError();
        return fail(TW_ERR_INVALID_ARG,
                    "chunk_tokens 0 reads the tensors in place: every tensor must be page-locked "
                    "host memory mapped into the device's address space");
    }
    // The alias rules were checked on the host addresses; a mapping keeps
    // each allocation's bytes contiguous and distinct allocations apart.
    Args c = a;
    c.partials = m_parts;
    c.out = m_out;
    c.residual = m_res;
    c.weight = m_weight;
    c.residual_out = m_res_out;
    c.host_direct = 1;
    return launch_range(c, *d, a.t0, a.t1, TW_PATH_CLUSTER, nullptr, stream);
}

int fused_from_host(const Args& a, void* workspace, size_t workspace_bytes,
                    int64_t chunk_tokens, void* stream) {
    int rc = check_args(a);
    if (rc != TW_OK) return rc;
    if (chunk_tokens == 0) return fused_in_place_from_host(a, stream);
    if (chunk_tokens < 0)
        return fail(TW_ERR_INVALID_ARG, "chunk_tokens %lld < 0", (long long)chunk_tokens);
    // A chunk never needs to be longer than the range; capped so, its bytes
    // stay within a buffer's (at most 2^48, checked above).
    const int64_t span = a.t1 - a.t0 > 1 ? a.t1 - a.t0 : 1;
    if (chunk_tokens > span) chunk_tokens = span;
    const int64_t rb = a.H * static_cast<int64_t>(elem_size(a.dtype));
    const size_t need = host_workspace_bytes(a.n_parts, a.n_out, rb, chunk_tokens);
    if (!workspace) return fail(TW_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(TW_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (workspace_bytes < need)
        return fail(TW_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    need);
    if (a.t0 == a.t1) return TW_OK;
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != TW_OK) return rc;
    // Every tensor must be page-locked host memory (the copies are async).
    const void* host_ptrs[TW_MAX_PARTS + TW_MAX_OUTS + 3];
    int n_ptrs = 0;
    for (int r = 0; r < a.n_parts; ++r) host_ptrs[n_ptrs++] = a.partials[r];
    for (int k = 0; k < a.n_out; ++k) host_ptrs[n_ptrs++] = a.out[k];
    host_ptrs[n_ptrs++] = a.residual;
    host_ptrs[n_ptrs++] = a.weight;
    host_ptrs[n_ptrs++] = a.residual_out;
    for (int i = 0; i < n_ptrs; ++i)
        if (!is_pinned_host(host_ptrs[i]))
            return fail(TW_ERR_INVALID_ARG, "tensor %d is not page-locked host memory", i);

    const HostCall hc{a.partials, a.n_parts, a.residual, a.weight, a.out, a.n_out,
                      a.residual_out, rb, a.t0, a.t1, chunk_tokens, workspace, stream};
    DeviceState& dev = *d;
    const LaunchChunk launch = [&](const void* const* parts, const void* residual,
                                   const void* weight, void* const* out, void* residual_out,
                                   int64_t n, cudaStream_t s) {
        Args c = a;
        c.partials = parts;
        c.residual = residual;
        c.weight = weight;
        c.out = out;
        c.residual_out = residual_out;
        c.T = n;
        c.t0 = 0;
        c.t1 = n;
        return launch_range(c, dev, 0, n, TW_PATH_AUTO, nullptr, s);
    };
    const char* what = nullptr;
    rc = host_pipeline(hc, launch, &what);
    if (rc > 0) return cuda_fail(static_cast<cudaError_t>(rc), what);
    return rc;
}

}  // namespace

int set_last_error(int code, const char* message) { return fail(code, "%s", message); }

int check_host_args(const void* const* partials, int n_parts, const void* residual,
                    const void* weight, void* const* out, int n_out, void* residual_out,
                    int64_t T, int64_t H, float eps, int64_t t0, int64_t t1, int max_sms,
                    int dtype) {
    const Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
                 T,        H,       eps,      t0,     t1,  max_sms, dtype};
    return check_args(a);
}

}  // namespace tw

using tw::Args;

extern "C" {

int tw_fused_reduce_add_rmsnorm_ex(const void* const* partials, int n_parts,
                                   const void* residual, const void* weight,
                                   void* const* out, int n_out, void* residual_out, int64_t T,
                                   int64_t H, float eps, int64_t t0, int64_t t1, int max_sms,
                                   void* stream, int dtype, int path, uint32_t* smid_log) {
    const Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
                 T,        H,       eps,      t0,     t1,  max_sms, dtype};
    return tw::fused(a, path, smid_log, stream);
}

int tw_fused_reduce_add_rmsnorm_colsplit(const void* const* partials, int n_parts,
                                         const void* residual, const void* weight,
                                         void* const* out, int n_out, void* residual_out,
                                         int64_t T, int64_t H, float eps, int64_t t0, int64_t t1,
                                         int max_sms, void* stream, int dtype) {
    Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
           T,        H,       eps,      t0,     t1,  max_sms, dtype};
    a.colsplit = 1;
    return tw::fused(a, TW_PATH_ROWS, nullptr, stream);
}

int tw_fused_reduce_add_rmsnorm_flags(const void* const* partials, int n_parts,
                                      const void* residual, const void* weight,
                                      void* const* out, int n_out, void* residual_out,
                                      int64_t T, int64_t H, float eps, int64_t t0, int64_t t1,
                                      int max_sms, void* stream, int dtype,
                                      const uint32_t* ready, int64_t block_tokens,
                                      uint32_t epoch) {
    if (!ready) return tw::fail(TW_ERR_INVALID_ARG, "ready is NULL");
    if ((reinterpret_cast<uintptr_t>(ready) & 3u) != 0)
        return tw::fail(TW_ERR_ALIGNMENT, "ready must be 4-byte aligned");
    if (block_tokens < 1)
        return tw::fail(TW_ERR_INVALID_ARG, "block_tokens %lld < 1", (long long)block_tokens);
    Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
           T,        H,       eps,      t0,     t1,  max_sms, dtype};
    a.ready = ready;
    a.block_tokens = block_tokens;
    a.epoch = epoch;
    return tw::fused(a, TW_PATH_ROWS, nullptr, stream);
}

int tw_fused_reduce_add_rmsnorm(const void* const* partials, int n_parts, const void* residual,
                                const void* weight, void* const* out, int n_out,
                                void* residual_out, int64_t T, int64_t H, float eps, int64_t t0,
                                int64_t t1, int max_sms, void* stream, int dtype) {
    return tw_fused_reduce_add_rmsnorm_ex(partials, n_parts, residual, weight, out, n_out,
                                          residual_out, T, H, eps, t0, t1, max_sms, stream,
                                          dtype, TW_PATH_AUTO, nullptr);
}

int tw_fused_reduce_add_rmsnorm_bf16(const void* const* partials, int n_parts,
                                     const void* residual, const void* weight,
                                     void* const* out, int n_out, void* residual_out,
                                     int64_t T, int64_t H, float eps, int64_t t0, int64_t t1,
                                     int max_sms, void* stream) {
    return tw_fused_reduce_add_rmsnorm(partials, n_parts, residual, weight, out, n_out,
                                       residual_out, T, H, eps, t0, t1, max_sms, stream,
                                       TW_BF16);
}

int tw_fused_reduce_add_rmsnorm_f32(const void* const* partials, int n_parts,
                                    const void* residual, const void* weight, void* const* out,
                                    int n_out, void* residual_out, int64_t T, int64_t H,
                                    float eps, int64_t t0, int64_t t1, int max_sms,
                                    void* stream) {
    return tw_fused_reduce_add_rmsnorm(partials, n_parts, residual, weight, out, n_out,
                                       residual_out, T, H, eps, t0, t1, max_sms, stream, TW_F32);
}

int tw_split_launch(const void* const* partials, int n_parts, const void* residual,
                    const void* weight, void* const* out, int n_out, void* residual_out,
                    int64_t T, int64_t H, float eps, int64_t t_split, int max_sms, void* s0,
                    void* s1, int dtype) {
    const Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
                 T,        H,       eps,      0,      T,   max_sms, dtype};
    int rc = tw::check_args(a);
    if (rc != TW_OK) return rc;
    if (t_split > T)
        return tw::fail(TW_ERR_INVALID_ARG, "t_split %lld > T %lld", (long long)t_split,
                        (long long)T);
    if (T == 0) return TW_OK;
    tw::DeviceState* d = nullptr;
    if ((rc = tw::device_state(&d)) != TW_OK) return rc;
    if (t_split < 0) {
        // Wave-aware default ("Der intelligente Split" names the idea, no
        // formula): T/2 moved to the nearest whole number of waves of the
        // first chunk's grid (one token per CTA per wave), so that chunk
        // ends without a partial last wave.
        const int64_t w = max_sms < d->sm_count ? max_sms : d->sm_count;
        t_split = T / 2;
        if (T >= 2 * w) t_split = (T / 2 + w / 2) / w * w;
    }

    cudaStream_t st0 = static_cast<cudaStream_t>(s0), st1 = static_cast<cudaStream_t>(s1);
    std::lock_guard<std::mutex> lock(d->split_mu);
    cudaError_t e;
    if ((e = cudaEventRecord(d->fork, st0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st1, d->fork, 0)) != cudaSuccess)
        return tw::cuda_fail(e, "fork");
    if (t_split > 0 &&
        (rc = tw::launch_range(a, *d, 0, t_split, TW_PATH_ROWS, nullptr, s0)) != TW_OK)
        return rc;
    if (t_split < T &&
        (rc = tw::launch_range(a, *d, t_split, T, TW_PATH_ROWS, nullptr, s1)) != TW_OK)
        return rc;
    if ((e = cudaEventRecord(d->join, st1)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st0, d->join, 0)) != cudaSuccess)
        return tw::cuda_fail(e, "join");
    return TW_OK;
}

int tw_host_workspace_bytes(int n_parts, int n_out, int64_t H, int64_t chunk_tokens, int dtype,
                            size_t* bytes) {
    if (!bytes || n_parts < 1 || n_parts > TW_MAX_PARTS || n_out < 1 || n_out > TW_MAX_OUTS ||
        H < 1 || H > (dtype == TW_BF16 ? TW_MAX_H_BF16 : TW_MAX_H_F32) || chunk_tokens < 1 ||
        (dtype != TW_BF16 && dtype != TW_F32))
        return tw::fail(TW_ERR_INVALID_ARG, "invalid workspace query");
    const int64_t rb = H * static_cast<int64_t>(tw::elem_size(dtype));
    // A chunk buffer is at most 2^48 bytes (a device address range), so the
    // size arithmetic below cannot overflow.
    if (chunk_tokens > (int64_t{1} << 48) / rb)
        return tw::fail(TW_ERR_INVALID_ARG, "chunks of %lld tokens of %lld bytes exceed 2^48 bytes",
                        (long long)chunk_tokens, (long long)rb);
    *bytes = tw::host_workspace_bytes(n_parts, n_out, rb, chunk_tokens);
    return TW_OK;
}

int tw_fused_reduce_add_rmsnorm_host(const void* const* partials, int n_parts,
                                     const void* residual, const void* weight, void* const* out,
                                     int n_out, void* residual_out, int64_t T, int64_t H,
                                     float eps, int64_t t0, int64_t t1, int max_sms,
                                     void* workspace, size_t workspace_bytes,
                                     int64_t chunk_tokens, void* stream, int dtype) {
    const Args a{partials, n_parts, residual, weight, out, n_out, residual_out,
                 T,        H,       eps,      t0,     t1,  max_sms, dtype};
    return tw::fused_from_host(a, workspace, workspace_bytes, chunk_tokens, stream);
}

int tw_device_status(int clear) {
    unsigned int word = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&word, tw::g_status_word, sizeof(word));
    if (e != cudaSuccess) return tw::cuda_fail(e, "cudaMemcpyFromSymbol"), -1;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(tw::g_status_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return tw::cuda_fail(e, "cudaMemcpyToSymbol"), -1;
    }
    return static_cast<int>(word);
}

const char* tw_last_error_string(void) { return tw::t_last_error.c_str(); }

int tw_version(void) { return TW_VERSION; }

}  // extern "C"
