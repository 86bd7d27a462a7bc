// tw_rows.cu -- the rows kernel: persistent CTAs, one token per CTA at a time.
//
// Per token t in [t0, t1) and feature h ("TokenWeave 策略详解", §1 背景 and
// §5 融合内核):
//   x = (sum_r partials[r][t,h]) + residual[t,h]      fp32, ranks in order
//   residual_out[t,h] = x
//   inv = 1 / sqrt(mean_h x^2 + eps)
//   out[k][t,h] = x * inv * weight[h]                 for every destination k
//
// Layout of the work: a token row of R = N + 1 input rows (the N partials and
// the residual) is cut into chunks of kChunkBytes per row.  One elected thread
// of the producer warp streams chunks into a ring of shared-memory stages with
// 1-D bulk async copies (cp.async.bulk, no tensor map, no multicast), each
// stage tracked by a "full" mbarrier (transaction bytes) and an "empty"
// mbarrier (one arrival per consumer warp).  The 256 consumer threads own one
// 16-byte vector of every chunk: they sum the staged rows in fp32, store
// residual_out at once, keep x in registers, and after the token's last chunk
// reduce the sum of squares (warp shuffle, then the 8 warp totals through
// shared memory behind one named barrier) and store the weighted result to
// every gather destination.  The N-way sum happens while the data streams
// through shared memory, the counterpart of the pages' sum-at-load.
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

template <typename T, int NC>
__global__ void __launch_bounds__(kRowsThreads + 32, 1)
    rows_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    using V = Vec<T>;
    constexpr int E = V::kElems;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    const int R = p.n_parts + 1;
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
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        if (p.smid_log) p.smid_log[blockIdx.x] = sm_id();
        mbar_init_fence();
    }
    __syncthreads();

    const int64_t first = p.t0 + blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t rb = p.row_bytes;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer ---
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0;
        for (int64_t t = first; t < p.t1; t += stride) {
            bool stop = false;
            for (int c = 0; c < NC; ++c, ++it) {
                const uint32_t s = it % S;
                if (*abort_flag ||
                    (it >= S && !mbar_wait(empty0 + 8 * s, ((it / S) - 1) & 1, abort_flag))) {
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
                for (int r = 0; r < p.n_parts; ++r, dst += kChunkBytes)
                    bulk_g2s(dst, static_cast<const char*>(p.partials[r]) + src_off, bytes, bar,
                             pol);
                bulk_g2s(dst, static_cast<const char*>(p.residual) + src_off, bytes, bar, pol);
            }
            if (stop) break;
        }
        // Drain: the copies of the last S issued stages must have landed before
        // this CTA may exit (bounded, also on the give-up path).
        const uint32_t lo = it > S ? it - S : 0;
        for (uint32_t j = lo; j < it; ++j)
            if (!mbar_wait(full0 + 8 * (j % S), (j / S) & 1, nullptr)) atomicOr(p.status, 2u);
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int64_t nvec = rb / 16;
    uint4 wv[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const int64_t v = static_cast<int64_t>(j) * kRowsThreads + tid;
        wv[j] = v < nvec ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                         : make_uint4(0, 0, 0, 0);
    }

    uint32_t it = 0;
    int red_buf = 0;
    bool alive = true;
    for (int64_t t = first; t < p.t1; t += stride) {
        float x[NC][E];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j, ++it) {
            const uint32_t s = it % S;
            if (alive && !mbar_wait(full0 + 8 * s, (it / S) & 1, abort_flag)) {
                give_up(p, abort_flag);
                alive = false;
            }
            const int64_t v = static_cast<int64_t>(j) * kRowsThreads + tid;
            if (v < nvec) {
                const unsigned char* src = ring + s * stage_bytes + tid * 16;
                float acc[E];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = 0.f;
                for (int r = 0; r < p.n_parts; ++r) {
                    float f[E];
                    V::to_float(*reinterpret_cast<const uint4*>(src + r * kChunkBytes), f);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] += f[e];
                }
                float f[E];
                V::to_float(*reinterpret_cast<const uint4*>(src + p.n_parts * kChunkBytes), f);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    x[j][e] = acc[e] + f[e];
                    ss = fmaf(x[j][e], x[j][e], ss);
                }
                if (alive)
                    st_global_cs(static_cast<char*>(p.residual_out) + t * rb + v * 16,
                                 V::from_float(x[j]));
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[j][e] = 0.f;
            }
            __syncwarp();
            if (alive && lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // Sum of squares over the token: warp shuffle, then the warp totals.
        ss = warp_sum(ss);
        if (lane == 0) red[red_buf * kConsumerWarps + warp] = ss;
        named_barrier(1, kRowsThreads);
        float total = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) total += red[red_buf * kConsumerWarps + w];
        red_buf ^= 1;
        const float inv = rsqrtf(total * p.inv_H + p.eps);

#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int64_t v = static_cast<int64_t>(j) * kRowsThreads + tid;
            if (v < nvec && alive) {
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

size_t rows_smem_bytes(int n_parts, int stages) {
    return static_cast<size_t>(kRingOff) +
           static_cast<size_t>(stages) * static_cast<size_t>(n_parts + 1) * kChunkBytes;
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

int launch_rows(const Params& p, int dtype, int grid, size_t smem_bytes, void* stream) {
    void* fn = rows_kernel_for(dtype, p.n_chunks);
    if (!fn) return static_cast<int>(cudaErrorInvalidValue);
    void* args[] = {const_cast<Params*>(&p)};
    return static_cast<int>(cudaLaunchKernel(fn, dim3(grid), dim3(kRowsThreads + 32), args,
                                             smem_bytes, static_cast<cudaStream_t>(stream)));
}

}  // namespace tw
