/*
 * tw.h -- C ABI of libtw.so: TokenWeave's fused reduce + residual add +
 * RMSNorm, recast for one GB300 (sm_103a) whose HBM holds all N rank partials.
 *
 * What it computes, per token t in [t0, t1) and feature h in [0, H):
 *
 *   x[t,h]            = (sum_{r=0}^{N-1} partials[r][t,h]) + residual[t,h]
 *   residual_out[t,h] = x[t,h]                                 rounded to dtype
 *   rms[t]            = sqrt( (1/H) * sum_h x[t,h]^2 + eps )
 *   out[k][t,h]       = x[t,h] / rms[t] * weight[h]   for k in [0, n_out), rounded to dtype
 *
 * Sources (page title, section):
 *   "TokenWeave 策略详解：以大模型推理为例", §1 背景: the layer output is
 *       RMSNorm(residual + allreduce_output) * weight, per token over all H
 *       features; the AllReduce is the sum of the rank partials.
 *   same page, §2 核心思想 and §3.2-3.4: the reordered ReduceScatter on token
 *       boundaries -> residual add -> RMSNorm -> AllGather; here the token
 *       range [t0, t1) is one rank's slice and the n_out destinations stand in
 *       for the AllGather buffers.
 *   same page, §5 融合内核: one launch, the sum taken at load time, residual
 *       and variance in registers, the result stored straight to the gather
 *       destinations.
 *   "TokenWeave: Efficient Compute-Communication Overlap for Distributed LLM
 *       Inference" (gist.science summary), "Der intelligente Split" and
 *       "Der Fused Kernel": a two-chunk token split run on two streams, and a
 *       fused kernel held to a small SM budget.
 * Readings where the pages are silent: eps inside the square root; no bias and
 * no (1 + w) offset; fp32 accumulation, the partials summed in rank order and
 * the residual added after them; the norm uses the fp32 x, not its rounded
 * copy; rounding to bf16 is round-to-nearest-even.
 *
 * Conventions for every entry point:
 *   - Pointers named partials/out are HOST arrays of DEVICE pointers (read
 *     during the call only).  Every other data pointer is a DEVICE pointer on
 *     the current CUDA device.  The caller owns all memory; the library
 *     allocates no device memory per call.
 *   - Tensors are dense row-major: partials[r], residual, out[k] and
 *     residual_out are [T, H] with row stride H elements; weight is [H].  All
 *     share one dtype (tw_dtype).
 *   - Only rows [t0, t1) of residual_out and of every out[k] are written; no
 *     other byte of any buffer is touched.  t0 == t1 returns TW_OK with no
 *     launch.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  A status other than TW_OK means nothing was launched.
 *     Faults after launch surface through the stream like any CUDA error.
 *     A launch whose max_sms covers every SM is a programmatic dependent
 *     launch: it may start while the previous kernel on the stream drains,
 *     but touches no global memory before that kernel has completed.
 *   - Argument rules, checked on the host before any CUDA call:
 *       partials/out arrays and every pointer in them non-NULL;
 *       1 <= n_parts <= TW_MAX_PARTS, 1 <= n_out <= TW_MAX_OUTS;
 *       T >= 0, 1 <= H <= TW_MAX_H(dtype), 0 <= t0 <= t1 <= T, and a
 *       buffer's T*H*size bytes fit in 2^48 (a device address range);
 *       eps finite and >= 0; max_sms >= 1 (values above the SM count clamp);
 *       H * sizeof(dtype) a multiple of 16 and every pointer 16-byte aligned
 *       (else TW_ERR_ALIGNMENT);
 *       residual_out may equal residual exactly (in place); any other overlap
 *       of an output with an input or with another output is TW_ERR_ALIAS
 *       (checked on the byte ranges [ptr, ptr + T*H*size)).
 *   - Errors: the return value is a tw_status; tw_last_error_string() gives a
 *     message for the calling thread's last failure.
 *   - Thread safety: calls from several host threads are safe; per-device state
 *     (SM count, fork/join events) is created once under a lock.
 */
#ifndef TW_H
#define TW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TW_VERSION 10100 /* 1.1.0: tw_set_ready, in-place host mode, claimed units */

#define TW_MAX_PARTS 16
#define TW_MAX_OUTS 8
/* Largest hidden size: 16384 bf16 or 8192 fp32 features, 32 KB per row (the
 * rows kernel keeps one token's fp32 x in registers, 32 floats per thread over
 * 512 threads). */
#define TW_MAX_H_BF16 16384
#define TW_MAX_H_F32 8192

typedef enum { TW_BF16 = 0, TW_F32 = 1 } tw_dtype;

typedef enum {
    TW_OK = 0,
    TW_ERR_INVALID_ARG = -1,
    TW_ERR_ALIGNMENT = -2,
    TW_ERR_ALIAS = -3,
    TW_ERR_CUDA = -4,
    TW_ERR_UNSUPPORTED = -5
} tw_status;

/* Kernel choice for tw_fused_reduce_add_rmsnorm_ex. */
typedef enum {
    TW_PATH_AUTO = 0,  /* cluster kernel for ranges of at most 128 tokens whose
                          clusters (one per token) can all run at once on the
                          device, when the row fits a cluster; rows kernel
                          otherwise */
    TW_PATH_ROWS = 1,  /* persistent CTAs, one token per CTA at a time, rows
                          staged into shared memory by bulk async copies */
    TW_PATH_WARP = 2,  /* one warp per token, no shared memory */
    TW_PATH_CLUSTER = 3 /* one thread-block cluster of C CTAs per token (C the
                           largest power of two <= min(8, max_sms)), the sum
                           of squares exchanged through distributed shared
                           memory; needs H * sizeof(dtype) <= C * 8 KB, else
                           TW_ERR_UNSUPPORTED.  Without a budget (max_sms at
                           least the SM count) CTAs may share SMs when the
                           clusters would not fit one CTA per SM. */
} tw_path;

/* The fused step on rows [t0, t1), bf16 tensors.  At most max_sms CTAs are
 * launched, each alone on its SM, so the kernel occupies at most max_sms SMs. */
int tw_fused_reduce_add_rmsnorm_bf16(const void* const* partials, int n_parts,
                                     const void* residual, const void* weight,
                                     void* const* out, int n_out,
                                     void* residual_out, int64_t T, int64_t H,
                                     float eps, int64_t t0, int64_t t1,
                                     int max_sms, void* stream);

/* Same, fp32 tensors. */
int tw_fused_reduce_add_rmsnorm_f32(const void* const* partials, int n_parts,
                                    const void* residual, const void* weight,
                                    void* const* out, int n_out,
                                    void* residual_out, int64_t T, int64_t H,
                                    float eps, int64_t t0, int64_t t1,
                                    int max_sms, void* stream);

/* Same, dtype given as a tw_dtype value. */
int tw_fused_reduce_add_rmsnorm(const void* const* partials, int n_parts,
                                const void* residual, const void* weight,
                                void* const* out, int n_out, void* residual_out,
                                int64_t T, int64_t H, float eps, int64_t t0,
                                int64_t t1, int max_sms, void* stream,
                                int dtype);

/* Same, with the kernel chosen explicitly (tw_path).  smid_log, when not NULL,
 * is a DEVICE array of at least max_sms uint32 entries; every CTA of the
 * launched kernel writes the id of the SM it ran on to smid_log[blockIdx.x]
 * (used to check the SM budget; entries of CTAs not launched are left
 * alone). */
int tw_fused_reduce_add_rmsnorm_ex(const void* const* partials, int n_parts,
                                   const void* residual, const void* weight,
                                   void* const* out, int n_out,
                                   void* residual_out, int64_t T, int64_t H,
                                   float eps, int64_t t0, int64_t t1,
                                   int max_sms, void* stream, int dtype,
                                   int path, uint32_t* smid_log);

/* Column-split partials ("TokenWeave 策略详解", appendix 实现方法：零填充 +
 * AllReduce 求和 and 数值示例): partial r is the zero-padded output of rank r,
 * nonzero only in columns [floor(r*H/n_parts), floor((r+1)*H/n_parts)), so the
 * sum over ranks is the concatenation of those slices.  Same computation and
 * arguments as tw_fused_reduce_add_rmsnorm, but only each rank's own slice is
 * read (the zero columns are never touched); the result is bit-identical to
 * the dense call on such inputs (adding zeros is exact).  Traffic per token:
 * (1 + 1 + n_out + 1) rows instead of (n_parts + 1 + n_out + 1).  Additional
 * rule: every slice boundary floor(r*H/n_parts) * sizeof(dtype) is a multiple
 * of 16 bytes (else TW_ERR_ALIGNMENT).  Runs on the rows kernel. */
int tw_fused_reduce_add_rmsnorm_colsplit(const void* const* partials, int n_parts,
                                         const void* residual, const void* weight,
                                         void* const* out, int n_out,
                                         void* residual_out, int64_t T, int64_t H,
                                         float eps, int64_t t0, int64_t t1,
                                         int max_sms, void* stream, int dtype);

/* Readiness flags (the FLUX notes' producer/consumer signals, WaitSignal and
 * SetSignal): the same step, but no row of token t is read before
 * ready[t / block_tokens] has reached `epoch` (compared as the signed 32-bit
 * difference ready - epoch >= 0, so epochs may wrap).  `ready` is a DEVICE
 * array of ceil(T / block_tokens) uint32 counters, 4-byte aligned, that a
 * producer raises (with release semantics) once the block's partials and
 * residual rows are written; it is read with acquire semantics at GPU scope.
 * Raising the counter per step (epoch = step number) reuses the array without
 * resetting it.  The wait is bounded: if a block's flag has not arrived
 * within about one second, the kernel stops reading and writing, sets the
 * value 4 in the device status word (tw_device_status) and returns; the rows
 * of the tokens that were waiting are then left unwritten (rows written before
 * are complete).  Runs on the rows kernel.
 * The producer's kernels must be loaded before this call starts waiting:
 * under CUDA's lazy module loading (the default) a kernel is loaded at its
 * first launch, and that load can wait for the kernels already running --
 * this one, spinning on the flags -- so the waits run out (status 4).  Launch
 * every producer kernel once beforehand; the library loads its own
 * (tw_set_ready's) when it sets up a device. */
int tw_fused_reduce_add_rmsnorm_flags(const void* const* partials, int n_parts,
                                      const void* residual, const void* weight,
                                      void* const* out, int n_out,
                                      void* residual_out, int64_t T, int64_t H,
                                      float eps, int64_t t0, int64_t t1,
                                      int max_sms, void* stream, int dtype,
                                      const uint32_t* ready,
                                      int64_t block_tokens, uint32_t epoch);

/* The producer side of the readiness flags (the FLUX notes' SetSignal):
 * after all work queued earlier on `stream` has completed -- the kernels or
 * copies that wrote the blocks' partial and residual rows -- set
 * ready[first_block + i] = epoch for i in [0, n_blocks), each with a release
 * store at GPU scope, so that tw_fused_reduce_add_rmsnorm_flags, whose
 * acquire read sees the flag, also sees those rows.  A plain store or memset
 * of the flags is a weak store and does not order the rows before the flag.
 * `ready` is a DEVICE array of uint32, 4-byte aligned; first_block and
 * n_blocks are in [0, 2^46]; n_blocks == 0 launches nothing.  Asynchronous
 * on `stream` (one small kernel). */
int tw_set_ready(uint32_t* ready, int64_t first_block, int64_t n_blocks,
                 uint32_t epoch, void* stream);

/* Two-chunk token split ("Der intelligente Split"): rows [0, t_split) run on
 * stream s0 and rows [t_split, T) on stream s1, each a rows-kernel launch with
 * its own budget of max_sms SMs (so up to 2*max_sms SMs while both run).
 * t_split < 0 picks T/2 moved to the nearest multiple of the first chunk's
 * grid, min(max_sms, SM count), when T is at least twice that (whole waves of
 * one token per CTA; the result does not depend on the split point).  s1
 * first waits for work already queued on s0, and
 * s0 is made to wait for the s1 chunk, so synchronising s0 alone covers both
 * chunks.  Same argument rules as above, with t_split <= T. */
int tw_split_launch(const void* const* partials, int n_parts,
                    const void* residual, const void* weight, void* const* out,
                    int n_out, void* residual_out, int64_t T, int64_t H,
                    float eps, int64_t t_split, int max_sms, void* s0, void* s1,
                    int dtype);

/* The fused step for tensors in page-locked HOST memory (cudaHostAlloc or
 * cudaHostRegister): partials, residual, weight, out and residual_out are host
 * pointers with the layout and rules above.
 * chunk_tokens == 0 (in place): one launch, on `stream`, whose kernel reads
 * the host tensors through their device mappings and stores straight into the
 * host outputs (plain loads and stores over the host link: the cluster
 * kernel).  Every tensor must be mapped into the device's address space
 * (cudaHostGetDevicePointer succeeds: all page-locked memory on a system with
 * unified addressing), else TW_ERR_INVALID_ARG; the row must fit the
 * cluster kernel (H * size <= 8 KB times the cluster size, 64 KB without a
 * budget), else TW_ERR_UNSUPPORTED.  `workspace` is not used (may be NULL).
 * chunk_tokens >= 1 (staged): only `workspace` is device memory,
 * at least tw_host_workspace_bytes() bytes, 256-byte aligned, owned by the
 * caller.  Rows [t0, t1) are moved in chunks of chunk_tokens tokens: the
 * host->device copies of one chunk overlap the kernel on the previous one, on
 * streams the library creates once per device.  When out and residual_out
 * are mapped into the device's address space (cudaHostGetDevicePointer
 * succeeds: all page-locked memory on a system with unified addressing) the
 * kernel stores the results straight into them; otherwise the results are
 * staged in the workspace and copied back on a third stream, overlapping the
 * following chunks.  `stream` orders the whole call (it waits for the last
 * kernel or copy back).  The host buffers and the workspace are in use until
 * the work on `stream` completes.  A chunk_tokens above t1 - t0 is cut to
 * t1 - t0 (the workspace is then checked against that chunk).  Returns
 * TW_ERR_INVALID_ARG if chunk_tokens < 0, a tensor is not page-locked host
 * memory or the workspace is too small. */
int tw_fused_reduce_add_rmsnorm_host(const void* const* partials, int n_parts,
                                     const void* residual, const void* weight,
                                     void* const* out, int n_out,
                                     void* residual_out, int64_t T, int64_t H,
                                     float eps, int64_t t0, int64_t t1,
                                     int max_sms, void* workspace,
                                     size_t workspace_bytes,
                                     int64_t chunk_tokens, void* stream,
                                     int dtype);

/* Device workspace bytes tw_fused_reduce_add_rmsnorm_host needs: the weight
 * and two slots of (n_parts + 1 + n_out + 1) chunk buffers, each rounded up to
 * 256 bytes.  TW_ERR_INVALID_ARG for arguments outside the rules above, or a
 * chunk buffer (chunk_tokens * H * size) above 2^48 bytes. */
int tw_host_workspace_bytes(int n_parts, int n_out, int64_t H,
                            int64_t chunk_tokens, int dtype, size_t* bytes);

/* Staging bytes the no-allocation entry point holds per GPU (see below). */
#define TW_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The host-buffer step of tw_fused_reduce_add_rmsnorm_host for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is a
 * convenience of this library.  Some callers cannot hand in a device
 * workspace: a host program that reaches the GPU only through this C ABI and
 * has no CUDA allocator of its own, a process whose device memory is all
 * reserved up front by a framework that gives out no raw buffers, or code
 * running where cudaMalloc is not allowed.  This entry point allocates
 * nothing: it stages the chunks in one device array of
 * TW_NOALLOC_SCRATCH_BYTES (16 MiB) that the library declares at file scope,
 * which every GPU that loads the library holds until the process exits.
 * Arguments are those of tw_fused_reduce_add_rmsnorm_host without the
 * workspace, checked first (t0 == t1 then returns TW_OK with no CUDA call);
 * chunk_tokens <= 0 picks the largest chunk, at most t1 - t0 tokens, whose
 * staging fits the array; a larger chunk_tokens is cut to t1 - t0; a chunk
 * whose staging needs more than the array holds is refused with
 * TW_ERR_UNSUPPORTED and a message naming both sizes (every row fits: one
 * token of the largest row and 25 buffers need under 2 MiB).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call on a device shares the one array and
 * it keeps the last call's contents; nothing in it needs to start at zero
 * (each chunk's staging is written before it is read).  Calls whose work
 * overlaps on the GPU (for instance issued on two streams without ordering
 * between them) race on the array: order them on one stream. */
int tw_fused_reduce_add_rmsnorm_host_noalloc(const void* const* partials,
                                             int n_parts, const void* residual,
                                             const void* weight,
                                             void* const* out, int n_out,
                                             void* residual_out, int64_t T,
                                             int64_t H, float eps, int64_t t0,
                                             int64_t t1, int max_sms,
                                             int64_t chunk_tokens, void* stream,
                                             int dtype);

/* Device-side status of the calling thread's current device: nonzero when a
 * kernel gave up on a bounded wait since the last clear, as an OR of 1 (an
 * async copy or stage that never completed), 2 (copies still in flight at
 * exit) and 4 (a readiness flag that never arrived).  Reading synchronises nothing; call it after the stream has
 * finished.  clear != 0 resets the word.  Returns -1 on a CUDA error. */
int tw_device_status(int clear);

/* Message for the calling thread's last failed call ("" if none). Never NULL. */
const char* tw_last_error_string(void);

/* TW_VERSION of the loaded library. */
int tw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TW_H */
