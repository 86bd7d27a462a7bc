// tw_cluster.cu -- the cluster kernel: one token per thread-block cluster, for
// decode-size ranges where a single warp or CTA per token leaves most of the
// GPU idle and a token's 100+ KB must arrive in one memory round trip.
//
// Same arithmetic as the other kernels ("TokenWeave 策略详解", §1 背景 and §5
// 融合内核): x = (sum_r partials[r]) + residual in fp32, ranks in order;
// residual_out = x; out[k] = x / sqrt(mean x^2 + eps) * weight.
//
// The C CTAs of a cluster split the token's columns into C contiguous slices.
// Each thread issues all N + 1 loads of its vectors at once, sums them, and
// the CTA's partial sum of squares is exchanged through distributed shared
// memory: every CTA writes its total into the shared memory of every CTA of
// the cluster, one cluster barrier makes them visible, and every thread adds
// the C totals in rank order from its own shared memory (so all CTAs get the
// same bits, and no CTA reads a peer's memory, so none has to wait for its
// peers before leaving).  No global scratch and no multicast.
#include "tw_device.cuh"

namespace tw {
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Full cluster barrier: release this CTA's shared-memory writes, acquire the
// peers'.  All CTAs of a cluster are co-scheduled, so it always completes.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cluster barrier in two halves: arrive (no ordering) early, wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Write a float into the shared memory of CTA `rank` of this cluster, at the
// same offset as `local` in this CTA.
__device__ __forceinline__ void st_peer_f32(float* local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// VPT: 16-byte vectors per thread and row; NP: partial rows held in
// registers at once (the smallest of 2, 4, 8, 16 that covers n_parts), so
// that a launch with few partials keeps few registers and more CTAs fit on
// an SM (N = 8 bf16 rows of 16 KB: 62 registers, 8 CTAs per SM, against 95
// and 5 when every launch reserved room for 16).
template <typename T, int VPT, int NP>
__global__ void __launch_bounds__(kClusterThreads)
    cluster_kernel(const __grid_constant__ Params p) {
    using V = Vec<T>;
    constexpr int E = V::kElems;
    constexpr int kWarps = kClusterThreads / 32;
    __shared__ float warp_part[kWarps];
    // cta_part[b][r]: CTA r's sum of squares of the token using buffer b,
    // written into every CTA of the cluster by CTA r itself.
    __shared__ float cta_part[2][kClusterMaxSize];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t crank = cluster_rank();
    const uint32_t csize = cluster_size();
    const int64_t nvec = p.row_bytes / 16;
    const int64_t per_cta = (nvec + csize - 1) / csize;
    const int64_t v_begin = static_cast<int64_t>(crank) * per_cta;
    const int64_t v_end = v_begin + per_cta < nvec ? v_begin + per_cta : nvec;
    // While the previous kernel of the stream drains (launches that may
    // overlap it only), warm L2 with this CTA's column slice of its first token (a prefetch only fills L2, where that
    // kernel's writes land too; the loads below come after the wait).
    if (tid == 0 && p.prefetch && v_begin < v_end) {
        const int64_t t = p.t0 + cluster_index();
        if (t < p.t1) {
            const int64_t off = t * p.row_bytes + v_begin * 16;
            const uint32_t bytes = static_cast<uint32_t>((v_end - v_begin) * 16);
            for (int r = 0; r < p.n_parts; ++r)
                bulk_prefetch_l2(static_cast<const char*>(p.partials[r]) + off, bytes);
            bulk_prefetch_l2(static_cast<const char*>(p.residual) + off, bytes);
        }
    }
    // Every CTA of the cluster must be running before any writes into its
    // shared memory: arrive now, wait just before the first such write (the
    // global loads of the first token hide the wait).
    cluster_arrive_relaxed();
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();
    bool peers_started = false;

    uint4 wv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int64_t v = v_begin + tid + k * kClusterThreads;
        wv[k] = v < v_end ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                          : make_uint4(0, 0, 0, 0);
    }

    int buf = 0;
    for (int64_t t = p.t0 + cluster_index(); t < p.t1; t += cluster_count()) {
        const int64_t row_off = t * p.row_bytes;
        // Warm L2 with this CTA's slice of the cluster's next token, so that
        // its loads overlap this token's reduction and stores.
        if (tid == 0 && p.prefetch && v_begin < v_end && t + cluster_count() < p.t1) {
            const int64_t off = (t + cluster_count()) * p.row_bytes + v_begin * 16;
            const uint32_t bytes = static_cast<uint32_t>((v_end - v_begin) * 16);
            for (int r = 0; r < p.n_parts; ++r)
                bulk_prefetch_l2(static_cast<const char*>(p.partials[r]) + off, bytes);
            bulk_prefetch_l2(static_cast<const char*>(p.residual) + off, bytes);
        }
        float x[VPT][E];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = v_begin + tid + k * kClusterThreads;
            const bool valid = v < v_end;
            uint4 raw[NP];
#pragma unroll
            for (int r = 0; r < NP; ++r)
                raw[r] = (valid && r < p.n_parts)
                             ? ld_global_nc(static_cast<const char*>(p.partials[r]) + row_off +
                                            v * 16)
                             : make_uint4(0, 0, 0, 0);
            const uint4 res = valid ? ld_global(static_cast<const char*>(p.residual) + row_off +
                                                v * 16)
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < E; ++e) x[k][e] = 0.f;
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                if (r < p.n_parts) {
                    float f[E];
                    V::to_float(raw[r], f);
#pragma unroll
                    for (int e = 0; e < E; ++e) x[k][e] += f[e];
                }
            }
            float f[E];
            V::to_float(res, f);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                x[k][e] += f[e];
                ss = fmaf(x[k][e], x[k][e], ss);
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) warp_part[warp] = ss;
        __syncthreads();
        if (!peers_started) {
            cluster_wait();
            peers_started = true;
        }
        // Thread r < C pushes this CTA's total into CTA r; after the barrier
        // every CTA holds all C totals locally and adds them in rank order
        // (the same bits everywhere).  A peer writes buffer `buf` again only
        // two tokens later, after the barrier of the next token, which this
        // CTA reaches only once it has read this one.
        if (tid < static_cast<int>(csize)) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += warp_part[w];
            st_peer_f32(&cta_part[buf][crank], static_cast<uint32_t>(tid), s);
        }
        cluster_sync();
        float total = 0.f;
        for (uint32_t r = 0; r < csize; ++r) total += cta_part[buf][r];
        buf ^= 1;
        const float inv = rsqrtf(total * p.inv_H + p.eps);

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = v_begin + tid + k * kClusterThreads;
            if (v < v_end) {
                const int64_t off = row_off + v * 16;
                st_global_cs(static_cast<char*>(p.residual_out) + off, V::from_float(x[k]));
                float w[E], y[E];
                V::to_float(wv[k], w);
#pragma unroll
                for (int e = 0; e < E; ++e) y[e] = (x[k][e] * inv) * w[e];
                const uint4 packed = V::from_float(y);
                for (int o = 0; o < p.n_out; ++o)
                    st_global_cs(static_cast<char*>(p.out[o]) + off, packed);
            }
        }
    }
    // A CTA with no token still completes the start-up barrier; after the
    // last token's barrier no CTA touches another's shared memory, so each
    // leaves as soon as its own stores are issued.
    if (!peers_started) cluster_wait();
}

template <typename T, int NP>
void* cluster_entry_np(int vpt) {
    switch (vpt) {
        case 1: return reinterpret_cast<void*>(&cluster_kernel<T, 1, NP>);
        case 2: return reinterpret_cast<void*>(&cluster_kernel<T, 2, NP>);
        case 4: return reinterpret_cast<void*>(&cluster_kernel<T, 4, NP>);
        default: return nullptr;
    }
}

template <typename T>
void* cluster_entry_for(int vpt, int np) {
    switch (np) {
        case 2: return cluster_entry_np<T, 2>(vpt);
        case 4: return cluster_entry_np<T, 4>(vpt);
        case 8: return cluster_entry_np<T, 8>(vpt);
        case 16: return cluster_entry_np<T, 16>(vpt);
        default: return nullptr;
    }
}

void* cluster_kernel_for(int dtype, int vpt, int np) {
    return dtype == TW_BF16 ? cluster_entry_for<__nv_bfloat16>(vpt, np)
                            : cluster_entry_for<float>(vpt, np);
}

}  // namespace

// Partials held in registers per thread: the smallest of 2, 4, 8, 16 that
// covers n_parts.
int cluster_np(int n_parts) {
    int np = 2;
    while (np < n_parts) np *= 2;
    return np;
}

int cluster_vectors_per_thread(int64_t row_bytes, int cluster) {
    const int64_t nvec = row_bytes / 16;
    const int64_t per_cta = (nvec + cluster - 1) / cluster;
    const int64_t need = (per_cta + kClusterThreads - 1) / kClusterThreads;
    for (int v = 1; v <= kClusterMaxVpt; v *= 2)
        if (v >= need) return v;
    return 0;
}

int cluster_set_attributes(int smem_optin) {
    // The kernel has a few bytes of static shared memory, so its dynamic
    // request stays at the exclusive-SM amount, not the full opt-in limit.
    if (smem_optin < kExclusiveSmemBytes + 1024) return static_cast<int>(cudaErrorInvalidValue);
    for (int dt = 0; dt < 2; ++dt)
        for (int v = 1; v <= kClusterMaxVpt; v *= 2)
            for (int np = 2; np <= 16; np *= 2) {
                cudaError_t e = cudaFuncSetAttribute(cluster_kernel_for(dt, v, np),
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     kExclusiveSmemBytes);
                if (e != cudaSuccess) return static_cast<int>(e);
            }
    return 0;
}

int cluster_max_active(int cluster, size_t smem_bytes, int dtype, int vpt, int np, int* n) {
    // The instantiations differ in registers (by vectors per thread and
    // partials held), so each is asked about separately.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return static_cast<int>(
        cudaOccupancyMaxActiveClusters(n, cluster_kernel_for(dtype, vpt, np), &cfg));
}

int launch_cluster(const Params& p, int dtype, int cluster, int n_clusters, size_t smem_bytes,
                   bool pdl, void* stream) {
    const int vpt = cluster_vectors_per_thread(p.row_bytes, cluster);
    void* fn = cluster_kernel_for(dtype, vpt, cluster_np(p.n_parts));
    if (!fn) return static_cast<int>(cudaErrorInvalidValue);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster * n_clusters));
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    void* args[] = {const_cast<Params*>(&p)};
    return static_cast<int>(cudaLaunchKernelExC(&cfg, fn, args));
}

}  // namespace tw
