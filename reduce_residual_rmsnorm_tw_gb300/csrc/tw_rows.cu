// tw_rows.cu -- the rows kernel: persistent CTAs, one token per CTA at a time.
//
// Per token t in [t0, t1) and feature h ("TokenWeave 策略详解", §1 背景 and
// §5 融合内核):
//   x = (sum_r partials[r][t,h]) + residual[t,h]      fp32, ranks in order
//   residual_out[t,h] = x
//   inv = 1 / sqrt(mean_h x^2 + eps)
//   out[k][t,h] = x * inv * weight[h]                 for every destination k
//
// Layout of the work: a token has R = N + 1 input rows (the N partials, then
// the residual), each H * b contiguous bytes.  A CTA's tokens t0 + b,
// t0 + b + grid, ... form one stream of rows, token after token.  One elected
// thread of the producer warp moves that stream, whole rows at a time, into a
// ring of shared-memory stages with 1-D bulk async copies (cp.async.bulk, one
// copy per row, no tensor map, no multicast); every stage holds the next
// `rows_per_stage` rows of the stream -- a stage may end one token and start
// the next -- and is tracked by a "full" mbarrier (transaction bytes) and an
// "empty" mbarrier (one arrival per consumer warp).  Large whole-row copies
// from several buffers in flight are what let one SM stream well above its
// share of HBM bandwidth, and uniform stages keep that true for any N and H.
// The 512 consumer threads own the 16-byte vectors tid, tid + 512, ... of a
// row: they add the staged rows into fp32 registers in row order (ranks
// first, residual last); when a token's residual row is in, they store
// residual_out, reduce the sum of squares (warp shuffle, then the 16 warp
// totals through shared memory behind one named barrier) and store the
// weighted result to every gather destination, then go on with the next
// token's rows.  The N-way sum happens while the data streams through shared
// memory, the counterpart of the pages' sum-at-load.
//
// Readiness flags (the FLUX notes' WaitSignal / SetSignal): with a `ready`
// array, the producer reads no row of token t before ready[t / block_tokens]
// has reached the call's epoch -- a bounded acquire wait; if a flag never
// arrives the CTA gives up (status bit 4), writes nothing more and exits.
//
// Column-split mode ("TokenWeave 策略详解", appendix 实现方法：零填充 +
// AllReduce 求和): partial r is zero outside its own column slice, so the sum
// is the concatenation of the slices.  The producer assembles one staged row
// from each rank's slice (one copy per rank); adding the zeros would change no
// bit (0 + p = p exactly), so the result equals the dense mode's, with
// (1 + 1 + n_out + 1) rows of traffic per token instead of (N + 1 + n_out + 1).
#include "tw_device.cuh"

namespace tw {
namespace {

constexpr int kConsumerWarps = kRowsThreads / 32;
constexpr int kFullOff = 0;
constexpr int kEmptyOff = 8 * kMaxStages;
constexpr int kRedOff = 16 * kMaxStages;
constexpr int kAbortOff = kRedOff + 2 * kConsumerWarps * 4;
constexpr int kRingOff = 1024;
static_assert(kAbortOff + 4 <= kRingOff, "shared header overflows");

__device__ __forceinline__ void give_up(const Params& p, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.status, 1u);
}

// Ring position: stage index and the parity of its current phase.
struct RingPos {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void advance(uint32_t S) {
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

template <typename T, int NV>
__global__ void __launch_bounds__(kRowsThreads + 32, 1)
    rows_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    using V = Vec<T>;
    constexpr int E = V::kElems;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    const int n_sum = p.colsplit ? 1 : p.n_parts;  // staged rows summed before the residual
    const int R = n_sum + 1;                        // staged rows per token
    const int G = p.rows_per_stage;
    const int64_t rb = p.row_bytes;
    const uint32_t stage_bytes = static_cast<uint32_t>(G * rb);
    const uint32_t full0 = smem_addr(smem + kFullOff);
    const uint32_t empty0 = smem_addr(smem + kEmptyOff);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
    const unsigned char* ring = smem + kRingOff;
    const uint32_t ring_addr = smem_addr(ring);

    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    // Everything above touched only shared memory; global memory may still be
    // in use by the previous kernel of the stream until this returns.
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();

    // This CTA's tokens and its row stream.
    const int64_t first = p.t0 + blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t my_tokens = first < p.t1 ? (p.t1 - first + stride - 1) / stride : 0;
    const int64_t total_rows = my_tokens * R;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer ---
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        RingPos pos;
        uint32_t issued = 0;
        int64_t tok = 0;            // token (index within this CTA) of the next row
        int g_next = 0;             // row within that token
        int64_t checked = -1;       // last token whose readiness flag was seen
        int64_t ready_block = -1;   // last flag block seen ready
        for (int64_t q0 = 0; q0 < total_rows; q0 += G, ++issued, pos.advance(S)) {
            const int n_rows = total_rows - q0 < G ? static_cast<int>(total_rows - q0) : G;
            if (p.ready) {
                // Every token that starts in this stage must be ready first.
                const int64_t last_tok = (q0 + n_rows - 1) / R;
                bool ok = true;
                for (int64_t i = checked + 1; i <= last_tok && ok; ++i) {
                    const int64_t b = (first + i * stride) / p.block_tokens;
                    if (b != ready_block) {
                        ok = flag_wait(p.ready + b, p.epoch, abort_flag);
                        ready_block = b;
                    }
                    checked = i;
                }
                if (!ok) {
                    give_up(p, abort_flag);
                    atomicOr(p.status, 4u);
                    break;
                }
            }
            const uint32_t s = pos.stage;
            if (*abort_flag ||
                (issued >= S && !mbar_wait(empty0 + 8 * s, pos.phase ^ 1u, abort_flag))) {
                give_up(p, abort_flag);
                break;
            }
            const uint32_t bar = full0 + 8 * s;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_rows * rb));
            uint32_t dst = ring_addr + s * stage_bytes;
            for (int k = 0; k < n_rows; ++k, dst += static_cast<uint32_t>(rb)) {
                const int64_t row_off = (first + tok * stride) * rb;
                if (g_next == n_sum) {
                    bulk_g2s(dst, static_cast<const char*>(p.residual) + row_off,
                             static_cast<uint32_t>(rb), bar, pol);
                } else if (p.colsplit) {
                    // One staged row from every rank's own column slice.
                    for (int r = 0; r < p.n_parts; ++r) {
                        const int64_t lo = p.col_lo[r], hi = p.col_lo[r + 1];
                        if (lo < hi)
                            bulk_g2s(dst + static_cast<uint32_t>(lo),
                                     static_cast<const char*>(p.partials[r]) + row_off + lo,
                                     static_cast<uint32_t>(hi - lo), bar, pol);
                    }
                } else {
                    bulk_g2s(dst, static_cast<const char*>(p.partials[g_next]) + row_off,
                             static_cast<uint32_t>(rb), bar, pol);
                }
                if (++g_next == R) {
                    g_next = 0;
                    ++tok;
                }
            }
        }
        // Drain: the copies of the last S issued stages must have landed before
        // this CTA may exit (bounded, also on the give-up path).  Walk back
        // from the last issued stage.
        RingPos back = pos;
        for (uint32_t k = 0; k < S && k < issued; ++k) {
            if (back.stage == 0) {
                back.stage = S - 1;
                back.phase ^= 1u;
            } else {
                --back.stage;
            }
            if (!mbar_wait(full0 + 8 * back.stage, back.phase, nullptr)) atomicOr(p.status, 2u);
        }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int64_t nvec = rb / 16;
    uint4 wv[NV];
    bool valid[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int64_t v = static_cast<int64_t>(j) * kRowsThreads + tid;
        valid[j] = v < nvec;
        wv[j] = valid[j] ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                         : make_uint4(0, 0, 0, 0);
    }

    RingPos pos;
    int red_buf = 0;
    bool alive = true;
    int64_t tok = 0;  // token (index within this CTA) being summed
    int g_cur = 0;    // its rows summed so far
    float x[NV][E];
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int e = 0; e < E; ++e) x[j][e] = 0.f;
    for (int64_t q0 = 0; q0 < total_rows; q0 += G, pos.advance(S)) {
        const int n_rows = total_rows - q0 < G ? static_cast<int>(total_rows - q0) : G;
        const uint32_t s = pos.stage;
        if (alive && !mbar_wait(full0 + 8 * s, pos.phase, abort_flag)) {
            give_up(p, abort_flag);
            alive = false;
        }
        const unsigned char* stage = ring + s * stage_bytes + tid * 16;
        for (int k = 0; k < n_rows; ++k) {
            const unsigned char* row = stage + k * rb;
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (valid[j])
                    add_vec(x[j], *reinterpret_cast<const uint4*>(row + j * kRowsThreads * 16),
                            static_cast<T*>(nullptr));
            if (k == n_rows - 1) {
                // The stage's rows are all in registers: hand it back to the
                // producer before any epilogue below.
                __syncwarp();
                if (alive && lane == 0) mbar_arrive(empty0 + 8 * s);
            }
            if (++g_cur < R) continue;
            // The token's residual row is in: store residual_out, reduce the
            // sum of squares over the token, store every destination.
            const int64_t t = first + tok * stride;
            float ss2[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (valid[j]) {
                    sum_squares<E>(ss2, x[j]);
                    if (alive)
                        st_global_cs(static_cast<char*>(p.residual_out) + t * rb +
                                         (static_cast<int64_t>(j) * kRowsThreads + tid) * 16,
                                     V::from_float(x[j]));
                }
            }
            const float ss = warp_sum(ss2[0] + ss2[1]);
            if (lane == 0) red[red_buf * kConsumerWarps + warp] = ss;
            named_barrier(1, kRowsThreads);
            float total = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) total += red[red_buf * kConsumerWarps + w];
            red_buf ^= 1;
            const float inv = rsqrtf(total * p.inv_H + p.eps);
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (valid[j] && alive) {
                    float w[E], y[E];
                    V::to_float(wv[j], w);
#pragma unroll
                    for (int e = 0; e < E; ++e) y[e] = (x[j][e] * inv) * w[e];
                    const uint4 packed = V::from_float(y);
                    const int64_t off = t * rb + (static_cast<int64_t>(j) * kRowsThreads + tid) * 16;
                    for (int o = 0; o < p.n_out; ++o)
                        st_global_cs(static_cast<char*>(p.out[o]) + off, packed);
                }
#pragma unroll
                for (int e = 0; e < E; ++e) x[j][e] = 0.f;
            }
            g_cur = 0;
            ++tok;
        }
    }
}

template <typename T>
void* rows_entry_for(int nv) {
    switch (nv) {
        case 1: return reinterpret_cast<void*>(&rows_kernel<T, 1>);
        case 2: return reinterpret_cast<void*>(&rows_kernel<T, 2>);
        case 3: return reinterpret_cast<void*>(&rows_kernel<T, 3>);
        case 4: return reinterpret_cast<void*>(&rows_kernel<T, 4>);
        default: return nullptr;
    }
}

void* rows_kernel_for(int dtype, int nv) {
    return dtype == TW_BF16 ? rows_entry_for<__nv_bfloat16>(nv) : rows_entry_for<float>(nv);
}

int rows_vectors_per_thread(int64_t row_bytes) {
    return static_cast<int>((row_bytes / 16 + kRowsThreads - 1) / kRowsThreads);
}

}  // namespace

size_t rows_smem_bytes(size_t stage_bytes, int stages) {
    return static_cast<size_t>(kRingOff) + static_cast<size_t>(stages) * stage_bytes;
}

int rows_set_smem_limit(int smem_optin) {
    for (int dt = 0; dt < 2; ++dt)
        for (int nv = 1; nv <= kRowsMaxVecs; ++nv) {
            cudaError_t e = cudaFuncSetAttribute(rows_kernel_for(dt, nv),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 smem_optin);
            if (e != cudaSuccess) return static_cast<int>(e);
        }
    return 0;
}

int launch_rows(const Params& p, int dtype, int grid, size_t smem_bytes, bool pdl,
                void* stream) {
    void* fn = rows_kernel_for(dtype, rows_vectors_per_thread(p.row_bytes));
    if (!fn) return static_cast<int>(cudaErrorInvalidValue);
    return launch_with_pdl(fn, p, grid, kRowsThreads + 32, smem_bytes, pdl, stream);
}

}  // namespace tw
