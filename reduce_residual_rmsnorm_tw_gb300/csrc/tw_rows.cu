// tw_rows.cu -- the rows kernel: persistent CTAs, one token per CTA at a time.
//
// Per token t in [t0, t1) and feature h ("TokenWeave 策略详解", §1 背景 and
// §5 融合内核):
//   x = (sum_r partials[r][t,h]) + residual[t,h]      fp32, ranks in order
//   residual_out[t,h] = x
//   inv = 1 / sqrt(mean_h x^2 + eps)
//   out[k][t,h] = x * inv * weight[h]                 for every destination k
//
// Layout of the work: a token's R = N + 1 input rows (the N partials and the
// residual) are cut into chunks of kChunkBytes per row.  One elected thread of
// the producer warp streams chunks into a ring of shared-memory stages with
// 1-D bulk async copies (cp.async.bulk, no tensor map, no multicast), each
// stage tracked by a "full" mbarrier (transaction bytes) and an "empty"
// mbarrier (one arrival per consuming warp).  Two consumer groups of 256
// threads take alternate chunks of each token (group g the chunks c = g mod 2),
// so two stages are being summed at any time.  A consumer thread owns one
// 16-byte vector of each of its chunks: it sums the staged rows in fp32 (ranks
// in order, residual last), stores residual_out at once, keeps x in
// registers, and after the token's last chunk the sum of squares goes through
// a warp shuffle and the 16 warp totals through shared memory behind one named
// barrier; then the weighted result is stored to every gather destination.
// The N-way sum happens while the data streams through shared memory, the
// counterpart of the pages' sum-at-load.
//
// Column-split mode ("TokenWeave 策略详解", appendix 实现方法：零填充 +
// AllReduce 求和): partial r is zero outside its own column slice, so the sum
// is the concatenation of the slices.  The producer copies only each rank's
// slice of a chunk into one staged row; adding the zeros would change no bit
// (0 + p = p exactly), so the result equals the dense mode's, with
// (1 + 1 + n_out + 1) rows of traffic per token instead of (N + 1 + n_out + 1).
#include "tw_device.cuh"

namespace tw {
namespace {

constexpr int kGroups = kRowsGroups;
constexpr int kGroupWarps = kRowsThreads / 32;
constexpr int kConsumerThreads = kGroups * kRowsThreads;
constexpr int kConsumerWarps = kConsumerThreads / 32;
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

template <typename T, int NC>
__global__ void __launch_bounds__(kConsumerThreads + 32, 1)
    rows_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    using V = Vec<T>;
    constexpr int E = V::kElems;
    constexpr int kSlots = (NC + kGroups - 1) / kGroups;  // chunks per thread and token

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    const int n_sum = p.colsplit ? 1 : p.n_parts;  // staged rows summed before the residual
    const int R = n_sum + 1;
    const uint32_t stage_bytes = static_cast<uint32_t>(R) * kChunkBytes;
    const uint32_t full0 = smem_addr(smem + kFullOff);
    const uint32_t empty0 = smem_addr(smem + kEmptyOff);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
    const unsigned char* ring = smem + kRingOff;
    const uint32_t ring_addr = smem_addr(ring);

    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kGroupWarps);
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

    const int64_t first = p.t0 + blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t rb = p.row_bytes;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer ---
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        RingPos pos;
        uint32_t issued = 0;
        bool stop = false;
        for (int64_t t = first; t < p.t1 && !stop; t += stride) {
            for (int c = 0; c < NC; ++c, ++issued, pos.advance(S)) {
                const uint32_t s = pos.stage;
                if (*abort_flag ||
                    (issued >= S && !mbar_wait(empty0 + 8 * s, pos.phase ^ 1u, abort_flag))) {
                    give_up(p, abort_flag);
                    stop = true;
                    break;
                }
                const int64_t off = static_cast<int64_t>(c) * kChunkBytes;
                const int64_t left = rb - off;
                const uint32_t bytes = left < kChunkBytes ? static_cast<uint32_t>(left)
                                                          : static_cast<uint32_t>(kChunkBytes);
                const uint32_t bar = full0 + 8 * s;
                mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(R));
                uint32_t dst = ring_addr + s * stage_bytes;
                const int64_t src_off = t * rb + off;
                if (p.colsplit) {
                    // Row 0 of the stage receives, from each rank, the part of
                    // its column slice that falls in this chunk.
                    for (int r = 0; r < p.n_parts; ++r) {
                        const int64_t lo = p.col_lo[r] > off ? p.col_lo[r] : off;
                        const int64_t end = off + bytes;
                        const int64_t hi = p.col_lo[r + 1] < end ? p.col_lo[r + 1] : end;
                        if (lo < hi)
                            bulk_g2s(dst + static_cast<uint32_t>(lo - off),
                                     static_cast<const char*>(p.partials[r]) + t * rb + lo,
                                     static_cast<uint32_t>(hi - lo), bar, pol);
                    }
                    dst += kChunkBytes;
                } else {
                    for (int r = 0; r < p.n_parts; ++r, dst += kChunkBytes)
                        bulk_g2s(dst, static_cast<const char*>(p.partials[r]) + src_off, bytes,
                                 bar, pol);
                }
                bulk_g2s(dst, static_cast<const char*>(p.residual) + src_off, bytes, bar, pol);
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
    const int group = warp / kGroupWarps;       // consumes chunks c with c % kGroups == group
    const int gtid = tid - group * kRowsThreads;  // 0 .. kRowsThreads-1 within the group
    const int64_t nvec = rb / 16;
    uint4 wv[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
        const int c = group + j * kGroups;
        const int64_t v = static_cast<int64_t>(c) * kRowsThreads + gtid;
        wv[j] = (c < NC && v < nvec) ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                                     : make_uint4(0, 0, 0, 0);
    }

    RingPos pos;
    int red_buf = 0;
    bool alive = true;
    for (int64_t t = first; t < p.t1; t += stride) {
        float x[kSlots][E];
        float ss2[2] = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            if (c % kGroups == group) {
                const int j = c / kGroups;
                const uint32_t s = pos.stage;
                if (alive && !mbar_wait(full0 + 8 * s, pos.phase, abort_flag)) {
                    give_up(p, abort_flag);
                    alive = false;
                }
                const int64_t v = static_cast<int64_t>(c) * kRowsThreads + gtid;
#pragma unroll
                for (int e = 0; e < E; ++e) x[j][e] = 0.f;
                if (v < nvec) {
                    const unsigned char* src = ring + s * stage_bytes + gtid * 16;
#pragma unroll 4
                    for (int r = 0; r < n_sum; ++r)
                        add_vec(x[j], *reinterpret_cast<const uint4*>(src + r * kChunkBytes),
                                static_cast<T*>(nullptr));
                    add_vec(x[j], *reinterpret_cast<const uint4*>(src + n_sum * kChunkBytes),
                            static_cast<T*>(nullptr));
                    sum_squares<E>(ss2, x[j]);
                    if (alive)
                        st_global_cs(static_cast<char*>(p.residual_out) + t * rb + v * 16,
                                     V::from_float(x[j]));
                }
                __syncwarp();
                if (alive && lane == 0) mbar_arrive(empty0 + 8 * s);
            }
            pos.advance(S);
        }
        // Sum of squares over the token: warp shuffle, then the warp totals.
        const float ss = warp_sum(ss2[0] + ss2[1]);
        if (lane == 0) red[red_buf * kConsumerWarps + warp] = ss;
        named_barrier(1, kConsumerThreads);
        float total = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) total += red[red_buf * kConsumerWarps + w];
        red_buf ^= 1;
        const float inv = rsqrtf(total * p.inv_H + p.eps);

#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
            const int c = group + j * kGroups;
            const int64_t v = static_cast<int64_t>(c) * kRowsThreads + gtid;
            if (c < NC && v < nvec && alive) {
                float w[E], y[E];
                V::to_float(wv[j], w);
#pragma unroll
                for (int e = 0; e < E; ++e) y[e] = (x[j][e] * inv) * w[e];
                const uint4 packed = V::from_float(y);
                for (int k = 0; k < p.n_out; ++k)
                    st_global_cs(static_cast<char*>(p.out[k]) + t * rb + v * 16, packed);
            }
        }
    }
}

template <typename T, int NC>
void* rows_entry() {
    return reinterpret_cast<void*>(&rows_kernel<T, NC>);
}

template <typename T>
void* rows_entry_for(int nc) {
    switch (nc) {
        case 1: return rows_entry<T, 1>();
        case 2: return rows_entry<T, 2>();
        case 3: return rows_entry<T, 3>();
        case 4: return rows_entry<T, 4>();
        case 5: return rows_entry<T, 5>();
        case 6: return rows_entry<T, 6>();
        case 7: return rows_entry<T, 7>();
        case 8: return rows_entry<T, 8>();
        default: return nullptr;
    }
}

void* rows_kernel_for(int dtype, int nc) {
    return dtype == TW_BF16 ? rows_entry_for<__nv_bfloat16>(nc) : rows_entry_for<float>(nc);
}

}  // namespace

int rows_staged_rows(int n_parts, int colsplit) { return colsplit ? 2 : n_parts + 1; }

size_t rows_smem_bytes(int staged_rows, int stages) {
    return static_cast<size_t>(kRingOff) +
           static_cast<size_t>(stages) * static_cast<size_t>(staged_rows) * kChunkBytes;
}

int rows_set_smem_limit(int smem_optin) {
    for (int dt = 0; dt < 2; ++dt)
        for (int nc = 1; nc <= kMaxChunks; ++nc) {
            cudaError_t e = cudaFuncSetAttribute(rows_kernel_for(dt, nc),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 smem_optin);
            if (e != cudaSuccess) return static_cast<int>(e);
        }
    return 0;
}

int launch_rows(const Params& p, int dtype, int grid, size_t smem_bytes, bool pdl,
                void* stream) {
    void* fn = rows_kernel_for(dtype, p.n_chunks);
    if (!fn) return static_cast<int>(cudaErrorInvalidValue);
    return launch_with_pdl(fn, p, grid, kConsumerThreads + 32, smem_bytes, pdl, stream);
}

}  // namespace tw
