// tw_warp.cu -- the warp kernel: one warp per token, for decode-size ranges.
//
// Same arithmetic as the rows kernel ("TokenWeave 策略详解", §1 背景 and §5
// 融合内核): x = (sum_r partials[r]) + residual in fp32, ranks in order;
// residual_out = x; out[k] = x / sqrt(mean x^2 + eps) * weight.
//
// A warp streams its token once with 16-byte loads, a step's loads for up to
// eight partial rows and the residual issued before any is used.  Pass 1
// accumulates the sum of squares, stores residual_out (each lane has read
// every row of the vectors it stores, so an in-place residual stays correct)
// and keeps x (fp32) in the warp's own shared memory; the warp-shuffle total
// gives 1/rms; pass 2 reads x back and stores every gather destination.  No
// block barrier is used.  Rows too long for four warps' x to fit the shared
// memory (bf16 rows above 28 KB) take the two-pass form: pass 2 streams the
// rows again (from L2) and recomputes x in the same order, bit-identical to
// pass 1, storing residual_out only then.
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

    // Whole steps (every lane's kLaneVecs vectors inside the row, the usual
    // case) skip the per-vector bounds checks; the byte offset is formed once.
    const bool whole = idx0 + (kLaneVecs - 1) * 32 < nvec;
    const int64_t off = row_off + idx0 * 16;
    for (int r0 = 0; r0 < p.n_parts; r0 += kPartGroup) {
        // Every load of the group -- and, with the last group, the residual's
        // -- is issued before any is used: one memory round trip per group.
        const bool last = r0 + kPartGroup >= p.n_parts;
        uint4 raw[kPartGroup][kLaneVecs];
        uint4 res[kLaneVecs];
#pragma unroll
        for (int q = 0; q < kPartGroup; ++q) {
            const int r = r0 + q < p.n_parts ? r0 + q : 0;  // any valid row when unused
            const char* src = static_cast<const char*>(p.partials[r]) + off;
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u)
                raw[q][u] = (r0 + q < p.n_parts && (whole || idx0 + u * 32 < nvec))
                                ? ld_global_nc(src + u * 32 * 16)
                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kLaneVecs; ++u)
            res[u] = (last && (whole || idx0 + u * 32 < nvec))
                         ? ld_global(static_cast<const char*>(p.residual) + off + u * 32 * 16)
                         : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < kPartGroup; ++q) {
            if (r0 + q < p.n_parts) {
#pragma unroll
                for (int u = 0; u < kLaneVecs; ++u)
                    add_vec(x[u], raw[q][u], static_cast<T*>(nullptr));
            }
        }
        if (last) {
            // The residual is added after every partial, as everywhere.
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u) add_vec(x[u], res[u], static_cast<T*>(nullptr));
        }
    }
}

// Shared memory one warp uses to keep its token's x (fp32) between the two
// passes: the row's vectors split in two halves of 16 bytes each (lane
// stride 16 bytes, so a warp's accesses are conflict-free).
__host__ __device__ __forceinline__ int64_t warp_x_bytes(int64_t row_bytes, int elem_bytes) {
    return (row_bytes / 16) * 16 * (4 / elem_bytes);
}

// STAGED: pass 1 also keeps x in the warp's shared memory and stores
// residual_out, and pass 2 reads x back instead of streaming the rows again.
template <typename T, bool STAGED>
__global__ void __launch_bounds__(kWarpTokensPerCta * 32)
    warp_kernel(const __grid_constant__ Params p) {
    using V = Vec<T>;
    constexpr int E = V::kElems;
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();
    grid_launch_dependents();
    if (threadIdx.x == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();

    const int64_t nvec = p.row_bytes / 16;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarpTokensPerCta;
    const int64_t step = 32 * kLaneVecs;
    // x of vector idx: xs[(h * nvec + idx)] for the halves h = 0, 1 (bf16:
    // 8 floats per vector, 4 in each half; fp32: 4 floats, all in half 0).
    float4* xs = reinterpret_cast<float4*>(
        smem + (threadIdx.x >> 5) * warp_x_bytes(p.row_bytes, static_cast<int>(sizeof(T))));
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
            if (STAGED) {
#pragma unroll
                for (int u = 0; u < kLaneVecs; ++u) {
                    const int64_t idx = base + lane + u * 32;
                    if (idx < nvec) {
                        // Every row of this token was read above (this lane's
                        // own vectors), so residual_out may overwrite an
                        // in-place residual now.
                        st_global_cs(static_cast<char*>(p.residual_out) + row_off + idx * 16,
                                     V::from_float(x[u]));
#pragma unroll
                        for (int h = 0; h < E / 4; ++h)
                            xs[h * nvec + idx] = make_float4(x[u][4 * h], x[u][4 * h + 1],
                                                             x[u][4 * h + 2], x[u][4 * h + 3]);
                    }
                }
            }
        }
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss * p.inv_H + p.eps);

        for (int64_t base = 0; base < nvec; base += step) {
            float x[kLaneVecs][E];
            if (STAGED) {
#pragma unroll
                for (int u = 0; u < kLaneVecs; ++u) {
                    const int64_t idx = base + lane + u * 32;
#pragma unroll
                    for (int h = 0; h < E / 4; ++h) {
                        const float4 q = idx < nvec ? xs[h * nvec + idx]
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                        x[u][4 * h] = q.x;
                        x[u][4 * h + 1] = q.y;
                        x[u][4 * h + 2] = q.z;
                        x[u][4 * h + 3] = q.w;
                    }
                }
            } else {
                token_x<T>(p, row_off, base + lane, nvec, x);
            }
#pragma unroll
            for (int u = 0; u < kLaneVecs; ++u) {
                const int64_t idx = base + lane + u * 32;
                if (idx < nvec) {
                    if (!STAGED)
                        st_global_cs(static_cast<char*>(p.residual_out) + row_off + idx * 16,
                                     V::from_float(x[u]));
                    float w[E], y[E];
                    V::to_float(ld_global_nc(static_cast<const char*>(p.weight) + idx * 16), w);
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        // (x * inv) * w two lanes at a time, each rounded as the
                        // scalar multiplies are.
                        asm("{\n\t.reg .b64 a, b, c;\n\t"
                            "mov.b64 a, {%2, %3};\n\t"
                            "mov.b64 b, {%4, %4};\n\t"
                            "mul.rn.f32x2 a, a, b;\n\t"
                            "mov.b64 c, {%5, %6};\n\t"
                            "mul.rn.f32x2 a, a, c;\n\t"
                            "mov.b64 {%0, %1}, a;\n\t}"
                            : "=f"(y[e]), "=f"(y[e + 1])
                            : "f"(x[u][e]), "f"(x[u][e + 1]), "f"(inv), "f"(w[e]), "f"(w[e + 1]));
                    }
                    const uint4 packed = V::from_float(y);
                    for (int k = 0; k < p.n_out; ++k)
                        st_global_cs(static_cast<char*>(p.out[k]) + row_off + idx * 16, packed);
                }
            }
        }
        // The next token's pass 1 overwrites xs: every lane must be done
        // reading it (each lane reads only what it wrote, but keep the warp
        // together).
        __syncwarp();
    }
}

void* warp_kernel_for(int dtype, bool staged) {
    if (dtype == TW_BF16)
        return staged ? reinterpret_cast<void*>(&warp_kernel<__nv_bfloat16, true>)
                      : reinterpret_cast<void*>(&warp_kernel<__nv_bfloat16, false>);
    return staged ? reinterpret_cast<void*>(&warp_kernel<float, true>)
                  : reinterpret_cast<void*>(&warp_kernel<float, false>);
}

}  // namespace

int warp_set_smem_limit(int smem_optin) {
    for (int dt = 0; dt < 2; ++dt)
        for (int staged = 0; staged < 2; ++staged) {
            cudaError_t e = cudaFuncSetAttribute(warp_kernel_for(dt, staged != 0),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 smem_optin);
            if (e != cudaSuccess) return static_cast<int>(e);
        }
    return 0;
}

size_t warp_stage_bytes(int64_t row_bytes, int dtype) {
    return static_cast<size_t>(kWarpTokensPerCta) *
           static_cast<size_t>(warp_x_bytes(row_bytes, dtype == TW_BF16 ? 2 : 4));
}

int launch_warp(const Params& p, int dtype, int grid, size_t smem_bytes, bool staged, bool pdl,
                void* stream) {
    return launch_with_pdl(warp_kernel_for(dtype, staged), p, grid, kWarpTokensPerCta * 32,
                           smem_bytes, pdl, stream);
}

}  // namespace tw
