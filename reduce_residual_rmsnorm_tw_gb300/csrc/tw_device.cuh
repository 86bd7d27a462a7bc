// tw_device.cuh -- device helpers for the sm_103a kernels: mbarrier and
// bulk-async-copy PTX, L2 cache policies, bounded waits, bf16/fp32 vector
// packing.  Everything here is written from the public PTX ISA description.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tw_internal.h"

namespace tw {

// ---------------------------------------------------------------- timers ---
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t id;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
    return id;
}

// Every wait on an mbarrier gives up after this long; a healthy pipeline
// stage completes in microseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false when
// the CTA is aborting (abort non-NULL and set by another thread) or after
// kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (global_timer_ns() - start > kWaitLimitNs) return false;
    }
}

// One acquire read of a readiness flag: has *flag reached `epoch` (compared
// wrap-safe as a signed difference)?
__device__ __forceinline__ bool flag_is_ready(const unsigned int* flag, unsigned int epoch) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return static_cast<int>(v - epoch) >= 0;
}

// Wait until *flag has reached `epoch` (compared wrap-safe as a signed
// difference), reading with acquire semantics at GPU scope, then order the
// async proxy (bulk copies) after it.  Returns false after kWaitLimitNs or
// when the CTA is aborting.
__device__ __forceinline__ bool flag_wait(const unsigned int* flag, unsigned int epoch,
                                          const volatile int* abort) {
    const uint64_t start = global_timer_ns();
    while (true) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (static_cast<int>(v - epoch) >= 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            return true;
        }
        if (abort && *abort) return false;
        if (global_timer_ns() - start > kWaitLimitNs) return false;
        __nanosleep(256);
    }
}

// ------------------------------------------------------ bulk async copy ---
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on
// `bar` as transaction bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  wait: block until the grids this launch
// depends on have completed and their memory is visible (a no-op when the
// launch had no programmatic dependency).  launch_dependents: allow the next
// grid of the stream to begin launching.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warm L2 with `bytes` bytes at `src` (a bulk prefetch: no data returns to
// the SM, nothing waits on it).  src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier over `threads` threads (a multiple of 32), id != 0.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the OR of `pred` over the `threads`
// participating threads (the same value in all of them).
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t threads, bool pred) {
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(any)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
        : "memory");
    return any != 0;
}

// ---------------------------------------------------- 16-byte vectors ---
// A 16-byte vector holds 8 bf16 or 4 fp32 elements.
template <typename T>
struct Vec;

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void to_float(const uint4& v, float* f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 from_float(const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Vec<float> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void to_float(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 from_float(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

// acc[e] += element e of the 16-byte vector v, in fp32 with one rounding per
// add (the same bits as widening the element and adding).  bf16 elements go
// through the mixed-precision add (the bf16 operand is widened exactly);
// fp32 pairs through the packed two-lane add.
__device__ __forceinline__ void add_vec(float (&acc)[8], const uint4& v, __nv_bfloat16*) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\t"
            "add.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "r"(w[i]));
}
__device__ __forceinline__ void add_vec(float (&acc)[4], const uint4& v, float*) {
    asm("{\n\t.reg .b64 a, b;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 a, a, b;\n\t"
        "mov.b64 {%0, %1}, a;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%6, %7};\n\t"
        "add.rn.f32x2 a, a, b;\n\t"
        "mov.b64 {%2, %3}, a;\n\t}"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// ss2 += x * x on two lanes at a time (packed fp32 FMA); the caller adds the
// two lanes at the end.
template <int E>
__device__ __forceinline__ void sum_squares(float (&ss2)[2], const float (&x)[E]) {
#pragma unroll
    for (int e = 0; e < E; e += 2)
        asm("{\n\t.reg .b64 a, s;\n\t"
            "mov.b64 a, {%2, %3};\n\t"
            "mov.b64 s, {%0, %1};\n\t"
            "fma.rn.f32x2 s, a, a, s;\n\t"
            "mov.b64 {%0, %1}, s;\n\t}"
            : "+f"(ss2[0]), "+f"(ss2[1])
            : "f"(x[e]), "f"(x[e + 1]));
}

// Streaming 16-byte global store (written once, not re-read by this kernel).
__device__ __forceinline__ void st_global_cs(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// Read-only 16-byte global load that does not allocate in L1.  Volatile so
// the compiler never hoists it out of the bounds check that guards it.
__device__ __forceinline__ uint4 ld_global_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Coherent 16-byte global load (used where the buffer may also be written by
// this kernel, e.g. a residual updated in place).
__device__ __forceinline__ uint4 ld_global(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Host side: launch fn(p) with the given shape, optionally with programmatic
// stream serialization (see grid_dependency_wait).  Returns a cudaError_t.
inline int launch_with_pdl(void* fn, const Params& p, int grid, int block, size_t smem_bytes,
                           bool pdl, void* stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {const_cast<Params*>(&p)};
    return static_cast<int>(cudaLaunchKernelExC(&cfg, fn, args));
}

}  // namespace tw
