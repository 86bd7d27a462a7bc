// tw_warp.cu -- the warp kernel: one warp per token, for decode-size ranges.
//
// Same arithmetic as the rows kernel ("TokenWeave 策略详解", §1 背景 and §5
// 融合内核): x = (sum_r partials[r]) + residual in fp32, ranks in order;
// residual_out = x; out[k] = x / sqrt(mean x^2 + eps) * weight.
//
// A warp streams its token twice with 16-byte loads, a step's loads for up to
// eight partial rows and the residual issued before any is used.  Pass 1 only
// accumulates
// the sum of squares (loads keep the default L2 policy, so the row stays in
// L2); the warp-shuffle total gives 1/rms.  Pass 2 recomputes x in the same
// order -- bit-identical to pass 1 -- and stores residual_out and every gather
// destination.  No shared memory and no block barrier are used; storing
// residual_out only in pass 2 keeps an in-place residual (residual_out ==
// residual) correct.
#include "tw_device.cuh"

namespace tw {
namespace {

constexpr int kLaneVecs = 4;    // 16-byte vectors per lane per step
constexpr int kPartGroup = 8;   // partial rows loaded together (the residual
                                // rides with the last group)

// x for the kLaneVecs vectors idx0 + u*32 of token row `row_off` (bytes).
// Vectors at or beyond nvec yield x = 0.
template <typename T>
__device__ __forceinline__ void token_x(const Params& p, int64_t row_off, int64_t idx0,
                                        int64_t nvec, float (&x)[kLaneVecs][Vec<T>::kElems]) {
    using V = Vec<T>;
    constexpr int E = V::kElems;
#pragma unroll
    for (int u = 0; u < kLaneVecs; ++u)
#pragma unroll
        for (int e = 0; e < E; ++e) x[u][e] = 0.f;

    for (int r0 = 0; r0 < p.n_parts; r0 += kPartGroup) {
        // Every load of the group -- and, with the last group, the residual's
        // -- is issued before any is used: one memory round trip per group.
        const bool last = r0 + kPartGroup >= p.n_parts;
        uint4 raw[kPartGroup][kLaneVecs];
        uint4 res[kLaneVecs];
#pragma unroll
        for (int q = 0; q < kPartGroup; ++q)
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u) {
                const int64_t idx = idx0 + u * 32;
                raw[q][u] = (r0 + q < p.n_parts && idx < nvec)
                                ? ld_global_nc(static_cast<const char*>(p.partials[r0 + q]) +
                                               row_off + idx * 16)
                                : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int u = 0; u < kLaneVecs; ++u) {
            const int64_t idx = idx0 + u * 32;
            res[u] = (last && idx < nvec)
                         ? ld_global(static_cast<const char*>(p.residual) + row_off + idx * 16)
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < kPartGroup; ++q) {
            if (r0 + q < p.n_parts) {
#pragma unroll
                for (int u = 0; u < kLaneVecs; ++u) {
                    float f[E];
                    V::to_float(raw[q][u], f);
#pragma unroll
                    for (int e = 0; e < E; ++e) x[u][e] += f[e];
                }
            }
        }
        if (last) {
            // The residual is added after every partial, as everywhere.
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u) {
                float f[E];
                V::to_float(res[u], f);
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] += f[e];
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kWarpTokensPerCta * 32)
    warp_kernel(const __grid_constant__ Params p) {
    using V = Vec<T>;
    constexpr int E = V::kElems;
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();

    const int64_t nvec = p.row_bytes / 16;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarpTokensPerCta;
    const int64_t step = 32 * kLaneVecs;
    for (int64_t t = p.t0 + static_cast<int64_t>(blockIdx.x) * kWarpTokensPerCta +
                     (threadIdx.x >> 5);
         t < p.t1; t += warps) {
        const int64_t row_off = t * p.row_bytes;

        float ss = 0.f;
        for (int64_t base = 0; base < nvec; base += step) {
            float x[kLaneVecs][E];
            token_x<T>(p, row_off, base + lane, nvec, x);
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u)
#pragma unroll
                for (int e = 0; e < E; ++e) ss = fmaf(x[u][e], x[u][e], ss);
        }
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss * p.inv_H + p.eps);

        for (int64_t base = 0; base < nvec; base += step) {
            float x[kLaneVecs][E];
            token_x<T>(p, row_off, base + lane, nvec, x);
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u) {
                const int64_t idx = base + lane + u * 32;
                if (idx < nvec) {
                    st_global_cs(static_cast<char*>(p.residual_out) + row_off + idx * 16,
                                 V::from_float(x[u]));
                    float w[E], y[E];
                    V::to_float(ld_global_nc(static_cast<const char*>(p.weight) + idx * 16), w);
#pragma unroll
                    for (int e = 0; e < E; ++e) y[e] = (x[u][e] * inv) * w[e];
                    const uint4 packed = V::from_float(y);
                    for (int k = 0; k < p.n_out; ++k)
                        st_global_cs(static_cast<char*>(p.out[k]) + row_off + idx * 16, packed);
                }
            }
        }
    }
}

void* warp_kernel_for(int dtype) {
    return dtype == TW_BF16 ? reinterpret_cast<void*>(&warp_kernel<__nv_bfloat16>)
                            : reinterpret_cast<void*>(&warp_kernel<float>);
}

}  // namespace

int warp_set_smem_limit(int smem_optin) {
    for (int dt = 0; dt < 2; ++dt) {
        cudaError_t e = cudaFuncSetAttribute(warp_kernel_for(dt),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_optin);
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    return 0;
}

int launch_warp(const Params& p, int dtype, int grid, size_t smem_bytes, bool pdl,
                void* stream) {
    return launch_with_pdl(warp_kernel_for(dtype), p, grid, kWarpTokensPerCta * 32, smem_bytes,
                           pdl, stream);
}

}  // namespace tw
