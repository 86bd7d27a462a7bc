// tw_rows.cu -- the rows kernel: persistent CTAs, one unit of tokens per CTA
// at a time.
//
// Per token t in [t0, t1) and feature h ("TokenWeave 策略详解", §1 背景 and
// §5 融合内核):
//   x = (sum_r partials[r][t,h]) + residual[t,h]      fp32, ranks in order
//   residual_out[t,h] = x
//   inv = 1 / sqrt(mean_h x^2 + eps)
//   out[k][t,h] = x * inv * weight[h]                 for every destination k
//
// Layout of the work: a token has R = N + 1 input rows (the N partials, then
// the residual), each H * b contiguous bytes.  CTAs take UNITS of U
// consecutive tokens (U = 1, 2 or 4, fixed per launch): with a fixed stride,
// or, in long launches, claimed one by one from a work counter (see the
// kernel).  Producer warps stream a unit's rows into a ring of shared-memory
// stages with 1-D bulk async copies (cp.async.bulk, no tensor map, no
// multicast): one copy per input buffer and unit covers the U consecutive
// rows of that buffer (contiguous in a row-major [T, H] tensor), so short
// rows still move in large copies.  A stage holds `rows_per_stage` such row
// groups of one unit (the host picks a whole unit when it fits, else an even
// split of its groups; a stage never crosses into the next unit) and is
// tracked by a "full" mbarrier (transaction bytes) and an "empty" mbarrier
// (one arrival per consumer warp).  The ring's stages are dealt round robin
// to `producers` warps (one elected lane each): the copy rate of one SM grows
// with the number of warps issuing copies (one issuing warp streamed ~36 GB/s
// of 16 KB copies whatever the ring depth, two ~69 GB/s), which is what bounds
// a CTA streaming alone on its SM under a small SM budget.  The 512 consumer
// threads own the 16-byte vectors tid, tid + 512, ... of a row: for each
// token of the unit they add the staged rows into fp32 registers in row order
// (ranks first, residual last); after the unit's last stage each token's sum
// of squares goes through a warp shuffle and the 16 warp totals of every
// token of the unit through shared memory behind ONE named barrier; then
// residual_out and the weighted result are stored for each token.  The N-way
// sum happens while the data streams through shared memory, the counterpart
// of the pages' sum-at-load.
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
// Warp totals of the sum of squares: double-buffered, U tokens x 16 warps,
// for each of the two consumer groups of the two-pipeline variant.
constexpr int kAbortOff = kRedOff + 2 * 2 * kRowsMaxUnit * kConsumerWarps * 4;
// Claimed-unit bookkeeping: the unit index each stage carries, the queue of
// claimed units producer 0 hands producer 1 ((unit, tag) pairs), and the last
// queue position producer 1 has read.
constexpr int kUnitQueue = 4;
constexpr int kStageUnitOff = kAbortOff + 8;
constexpr int kQueueOff = kStageUnitOff + 8 * kMaxStages;
constexpr int kSeenOff = kQueueOff + 16 * kUnitQueue;
constexpr int kRingOff = 2048;
// Tokens of its own a CTA prefetches into L2 before its first global read
// (three measured best), never more than kPrefetchMaxBytes, so the prefetch
// of a whole grid stays well inside L2.
constexpr int kPrefetchTokens = 3;
constexpr int64_t kPrefetchMaxBytes = 720 * 1024;
static_assert(kSeenOff + 8 <= kRingOff, "shared header overflows");

// Warm L2 with every input row of the n_tok tokens from t (bulk prefetches:
// nothing returns to the SM and nothing waits on them).
__device__ __forceinline__ void prefetch_tokens(const Params& p, int64_t t, int n_tok, int R,
                                                int n_sum) {
    const int64_t rb = p.row_bytes;
    const int64_t off = t * rb;
    const uint32_t bytes = static_cast<uint32_t>(n_tok * rb);
    for (int g = 0; g < R; ++g) {
        if (g == n_sum) {
            bulk_prefetch_l2(static_cast<const char*>(p.residual) + off, bytes);
        } else if (p.colsplit) {
            for (int j = 0; j < n_tok; ++j)
                for (int r = 0; r < p.n_parts; ++r)
                    if (p.col_lo[r] < p.col_lo[r + 1])
                        bulk_prefetch_l2(static_cast<const char*>(p.partials[r]) + off + j * rb +
                                             p.col_lo[r],
                                         static_cast<uint32_t>(p.col_lo[r + 1] - p.col_lo[r]));
        } else {
            bulk_prefetch_l2(static_cast<const char*>(p.partials[g]) + off, bytes);
        }
    }
}

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

constexpr int kRowsBlock = kRowsThreads + 32 * kRowsMaxProducers;

// Kernel variants (separate instantiations, so each carries only its code):
//   kFixed  -- CTA b takes units b, b + grid, b + 2 grid, ...
//   kClaim  -- CTA b's first unit is b; after that producer 0 claims units
//              from the launch's work counter (grid + an atomic increment),
//              one unit ahead, and hands them to producer 1 through a shared
//              queue; the first stage of each unit carries its index to the
//              consumers, and a stage holding -1 (no unit left) ends their
//              loop.  SMs that stream faster take more units (on a GB300
//              some groups of SMs stream ~10 % slower than the rest; with a
//              fixed share a long launch waits for them).
//   kFlags  -- the fixed schedule, each token read only once its readiness
//              flag is up.
// Every unit is processed exactly once, and a token's arithmetic does not
// depend on which CTA processes it.  U: tokens per unit (1, 2 or 4); NV:
// 16-byte vectors per consumer thread and row (U * NV <= kRowsMaxVecs).
constexpr int kFixed = 0, kClaim = 1, kFlags = 2;

template <typename T, int NV, int U, int MODE>
__global__ void __launch_bounds__(kRowsBlock, 1)
    rows_kernel(const __grid_constant__ Params p) {
    static_assert(U >= 1 && U <= kRowsMaxUnit && U * NV <= kRowsMaxVecs, "unit too large");
    static_assert(MODE != kFlags || U == 1, "readiness flags take one token per unit");
    constexpr bool FLAGS = MODE == kFlags;
    constexpr bool CLAIM = MODE == kClaim;
    extern __shared__ __align__(1024) unsigned char smem[];
    using V = Vec<T>;
    constexpr int E = V::kElems;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    const int n_sum = p.colsplit ? 1 : p.n_parts;  // rows summed before the residual
    const int R = n_sum + 1;                        // staged row groups per unit
    const int G = p.rows_per_stage;                 // row groups per stage
    const int stages_per_unit = (R + G - 1) / G;
    const int64_t rb = p.row_bytes;
    // A row group holds U consecutive token rows of one buffer (fewer in the
    // range's last unit, which leaves the rest of its slot unused).
    const uint32_t group_bytes = static_cast<uint32_t>(U * rb);
    const uint32_t stage_bytes = static_cast<uint32_t>(G) * group_bytes;
    const uint32_t full0 = smem_addr(smem + kFullOff);
    const uint32_t empty0 = smem_addr(smem + kEmptyOff);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
    volatile int64_t* stage_unit = reinterpret_cast<volatile int64_t*>(smem + kStageUnitOff);
    volatile int64_t* queue = reinterpret_cast<volatile int64_t*>(smem + kQueueOff);
    volatile int64_t* p1_seen = reinterpret_cast<volatile int64_t*>(smem + kSeenOff);
    const unsigned char* ring = smem + kRingOff;
    const uint32_t ring_addr = smem_addr(ring);
    const int64_t n_units = (p.t1 - p.t0 + U - 1) / U;

    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        if (CLAIM) {
            for (int q = 0; q < kUnitQueue; ++q) queue[2 * q + 1] = -1;  // nothing published
            *p1_seen = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();
    // While the previous kernel of the stream drains (launches that may
    // overlap it only), warm L2 with this CTA's first unit and the units the
    // fixed schedule gives it next (with claimed units some other CTA takes
    // those soon).  A prefetch only fills L2, which is where every write of
    // that kernel lands too, so data read after the wait below is current
    // even if the previous kernel writes these rows.  With readiness flags
    // only rows whose flag is already up are warmed (a raised flag means its
    // rows are final); the first token whose flag is not up ends the warming.
    if (warp == kConsumerWarps && lane == 0 && p.prefetch) {
        const int64_t unit_bytes = static_cast<int64_t>(R) * U * rb;
        int64_t n_pre = (kPrefetchTokens + U - 1) / U;  // units
        if (n_pre * unit_bytes > kPrefetchMaxBytes) n_pre = kPrefetchMaxBytes / unit_bytes;
        for (int64_t i = 0; i < n_pre; ++i) {
            const int64_t u = blockIdx.x + i * gridDim.x;
            if (u >= n_units) break;
            const int64_t t = p.t0 + u * U;
            if (FLAGS && !flag_is_ready(p.ready + t / p.block_tokens, p.epoch)) break;
            const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
            prefetch_tokens(p, t, n_tok, R, n_sum);
        }
    }
    // Everything above touched only shared memory (and L2 through prefetches);
    // global memory may still be in use by the previous kernel of the stream
    // until this returns.
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();

    if (warp >= kConsumerWarps) {
        // ----------------------------------------------------- producers ---
        // Producer `pw` issues the stages s with s % producers == pw (the
        // ring depth is a multiple of producers, so it owns the same slots
        // throughout); every producer walks the same stage sequence.
        const uint32_t P = static_cast<uint32_t>(p.producers);  // a power of two
        const uint32_t pw = static_cast<uint32_t>(warp - kConsumerWarps);
        if (lane != 0 || pw >= P) return;
        const uint64_t pol = policy_evict_first();
        RingPos pos;
        uint64_t issued = 0;  // stages of the sequence passed, by any producer
        bool stop = false;
        int64_t ready_block = -1;  // last flag block seen ready
        int64_t u = blockIdx.x;    // every CTA has a first unit (grid <= units)
        for (int64_t i = 0; !stop; ++i) {
            if (i > 0) {
                if (!CLAIM) {
                    u = blockIdx.x + i * gridDim.x;
                    if (u >= n_units) break;
                } else {
                    // Unit of position i, claimed by producer 0 during
                    // position i - 1 and published as (unit, tag i) in queue
                    // slot i % kUnitQueue; producer 1 waits (bounded) for it.
                    const int q = static_cast<int>(i % kUnitQueue);
                    if (pw != 0 && queue[2 * q + 1] != i) {
                        const uint64_t start = global_timer_ns();
                        while (queue[2 * q + 1] != i) {
                            if (*abort_flag || global_timer_ns() - start > kWaitLimitNs) {
                                give_up(p, abort_flag);
                                stop = true;
                                break;
                            }
                        }
                        if (stop) break;
                    }
                    __threadfence_block();
                    u = queue[2 * q];
                    if (pw != 0) *p1_seen = i;
                    if (u < 0) {
                        // No unit left: the owner of the next stage hands the
                        // consumers a stage holding -1 (an arrival without
                        // bytes), which ends their loop.
                        const uint32_t s = pos.stage;
                        if ((s & (P - 1)) == pw) {
                            if (issued >= S &&
                                !mbar_wait(empty0 + 8 * s, pos.phase ^ 1u, abort_flag)) {
                                give_up(p, abort_flag);
                            } else {
                                stage_unit[s] = -1;
                                mbar_arrive(full0 + 8 * s);
                            }
                        }
                        ++issued;
                        pos.advance(S);
                        break;
                    }
                }
            }
            // Producer 0 claims the unit of position i + 1 now and publishes
            // it once this unit's copies are issued, so the atomic's round
            // trip overlaps them.
            unsigned int claimed = 0;
            if (CLAIM && pw == 0) claimed = atomicAdd(p.work, 1u);
            const int64_t t = p.t0 + u * U;
            const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
            const uint32_t copy_bytes = static_cast<uint32_t>(n_tok * rb);
            const int64_t row_off = t * rb;
            for (int k = 0; k < stages_per_unit; ++k, ++issued, pos.advance(S)) {
                const uint32_t s = pos.stage;
                if ((s & (P - 1)) != pw) continue;
                if (FLAGS) {
                    const int64_t b = t / p.block_tokens;
                    if (b != ready_block) {
                        if (!flag_wait(p.ready + b, p.epoch, abort_flag)) {
                            give_up(p, abort_flag);
                            atomicOr(p.status, 4u);
                            stop = true;
                            break;
                        }
                        ready_block = b;
                    }
                }
                if (*abort_flag ||
                    (issued >= S && !mbar_wait(empty0 + 8 * s, pos.phase ^ 1u, abort_flag))) {
                    give_up(p, abort_flag);
                    stop = true;
                    break;
                }
                if (CLAIM && k == 0) stage_unit[s] = u;  // read by the consumers after the full wait
                const int g0 = k * G;
                const int g1 = g0 + G < R ? g0 + G : R;
                const uint32_t bar = full0 + 8 * s;
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>(g1 - g0) * copy_bytes);
                uint32_t dst = ring_addr + s * stage_bytes;
                for (int g = g0; g < g1; ++g, dst += group_bytes) {
                    if (g == n_sum) {
                        bulk_g2s(dst, static_cast<const char*>(p.residual) + row_off, copy_bytes,
                                 bar, pol);
                    } else if (p.colsplit) {
                        // One staged row per token from every rank's own
                        // column slice.
                        for (int j = 0; j < n_tok; ++j)
                            for (int r = 0; r < p.n_parts; ++r) {
                                const int64_t lo = p.col_lo[r], hi = p.col_lo[r + 1];
                                if (lo < hi)
                                    bulk_g2s(dst + static_cast<uint32_t>(j * rb + lo),
                                             static_cast<const char*>(p.partials[r]) + row_off +
                                                 j * rb + lo,
                                             static_cast<uint32_t>(hi - lo), bar, pol);
                            }
                    } else {
                        bulk_g2s(dst, static_cast<const char*>(p.partials[g]) + row_off,
                                 copy_bytes, bar, pol);
                    }
                }
            }
            if (CLAIM && pw == 0 && !stop) {
                // Publish position i + 1, at most kUnitQueue - 1 positions
                // ahead of producer 1's reads (p1_seen), so no queue slot is
                // overwritten before it is read.
                const int64_t next = static_cast<int64_t>(gridDim.x) + claimed;
                const int64_t j = i + 1;
                if (P > 1 && j - *p1_seen >= kUnitQueue) {
                    const uint64_t start = global_timer_ns();
                    while (j - *p1_seen >= kUnitQueue) {
                        if (*abort_flag || global_timer_ns() - start > kWaitLimitNs) {
                            give_up(p, abort_flag);
                            stop = true;
                            break;
                        }
                    }
                }
                if (!stop) {
                    const int q = static_cast<int>(j % kUnitQueue);
                    queue[2 * q] = next < n_units ? next : -1;
                    __threadfence_block();
                    queue[2 * q + 1] = j;
                }
            }
        }
        // The last CTA whose producer 0 is done claiming resets the counter
        // for the launch that next gets it (the host hands a counter to a
        // new launch only once the previous one has completed).
        if (CLAIM && pw == 0) {
            __threadfence();
            if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
                p.work[0] = 0;
                p.work[1] = 0;
            }
        }
        // Drain: this producer's copies into its slots must have landed before
        // the CTA may exit (bounded, also on the give-up path).  Walk back
        // over the last S stages of the sequence before the point where this
        // producer stopped: each of its slots appears once, at its last use.
        RingPos back = pos;
        for (uint32_t k = 0; k < S && k < issued; ++k) {
            if (back.stage == 0) {
                back.stage = S - 1;
                back.phase ^= 1u;
            } else {
                --back.stage;
            }
            if ((back.stage & (P - 1)) != pw) continue;
            if (!mbar_wait(full0 + 8 * back.stage, back.phase, nullptr)) atomicOr(p.status, 2u);
        }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int64_t nvec = rb / 16;
    uint4 wv[NV];
#pragma unroll
    for (int jj = 0; jj < NV; ++jj) {
        const int64_t v = static_cast<int64_t>(jj) * kRowsThreads + tid;
        wv[jj] = v < nvec ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                          : make_uint4(0, 0, 0, 0);
    }

    // Every consumer wait is bounded and every consumer passes the unit's
    // named barrier once per unit.  Fixed schedule: all consumers walk the
    // same units, and one that gave up keeps walking them (no waits, no
    // stores) so the barrier sequence stays whole.  Claimed units: the
    // barrier ORs the consumers' "stop" votes (a wait that gave up, or no
    // unit left), so all leave the loop at the same barrier.
    RingPos pos;
    int red_buf = 0;
    bool alive = true;
    for (int64_t i = 0;; ++i) {
        int64_t u = 0;
        if (!CLAIM) {
            u = blockIdx.x + i * gridDim.x;
            if (u >= n_units) break;
        }
        // The unit's first stage: with claimed units it carries the unit's
        // index (-1: none left).
        if (alive && !mbar_wait(full0 + 8 * pos.stage, pos.phase, abort_flag)) {
            give_up(p, abort_flag);
            alive = false;
        }
        bool none_left = false;
        if (CLAIM && alive) {
            u = stage_unit[pos.stage];
            none_left = u < 0;
            if (none_left) u = 0;
        }
        const int64_t t = p.t0 + u * U;
        const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
        float x[U][NV][E];
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int jj = 0; jj < NV; ++jj)
#pragma unroll
                for (int e = 0; e < E; ++e) x[j][jj][e] = 0.f;
        for (int k = 0; k < stages_per_unit; ++k, pos.advance(S)) {
            if (CLAIM && (!alive || none_left)) break;
            const uint32_t s = pos.stage;
            if (k > 0 && alive && !mbar_wait(full0 + 8 * s, pos.phase, abort_flag)) {
                give_up(p, abort_flag);
                alive = false;
            }
            const int g0 = k * G;
            const int g1 = g0 + G < R ? g0 + G : R;
            const unsigned char* stage = ring + s * stage_bytes + tid * 16;
            for (int g = g0; g < g1; ++g) {
                const unsigned char* group = stage + (g - g0) * group_bytes;
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    if (U == 1 || j < n_tok) {
                        const unsigned char* row = group + j * rb;
#pragma unroll
                        for (int jj = 0; jj < NV; ++jj)
                            if (static_cast<int64_t>(jj) * kRowsThreads + tid < nvec)
                                add_vec(x[j][jj],
                                        *reinterpret_cast<const uint4*>(row +
                                                                        jj * kRowsThreads * 16),
                                        static_cast<T*>(nullptr));
                    }
                }
            }
            __syncwarp();
            if (alive && lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // Every row of the unit is in, the residual last: reduce each token's
        // sum of squares (one barrier for the whole unit), then store.
        float* red_unit = red + red_buf * (U * kConsumerWarps);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            float ss2[2] = {0.f, 0.f};
#pragma unroll
            for (int jj = 0; jj < NV; ++jj)
                if (static_cast<int64_t>(jj) * kRowsThreads + tid < nvec)
                    sum_squares<E>(ss2, x[j][jj]);
            const float ss = warp_sum(ss2[0] + ss2[1]);
            if (lane == 0) red_unit[j * kConsumerWarps + warp] = ss;
        }
        if (CLAIM) {
            if (named_barrier_or(1, kRowsThreads, !alive || none_left)) break;
        } else {
            named_barrier(1, kRowsThreads);
        }
        red_buf ^= 1;
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (U > 1 && j >= n_tok) break;
            float total = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) total += red_unit[j * kConsumerWarps + w];
            const float inv = rsqrtf(total * p.inv_H + p.eps);
            const int64_t row_off = (t + j) * rb;
#pragma unroll
            for (int jj = 0; jj < NV; ++jj) {
                const int64_t v = static_cast<int64_t>(jj) * kRowsThreads + tid;
                if (v < nvec && alive) {
                    st_global_cs(static_cast<char*>(p.residual_out) + row_off + v * 16,
                                 V::from_float(x[j][jj]));
                    float w[E], y[E];
                    V::to_float(wv[jj], w);
#pragma unroll
                    for (int e = 0; e < E; ++e) y[e] = (x[j][jj][e] * inv) * w[e];
                    const uint4 packed = V::from_float(y);
                    for (int k = 0; k < p.n_out; ++k)
                        st_global_cs(static_cast<char*>(p.out[k]) + row_off + v * 16, packed);
                }
            }
        }
    }
}

template <typename T, int NV, int U, int MODE>
void* rows_fn() {
    return reinterpret_cast<void*>(&rows_kernel<T, NV, U, MODE>);
}

// The instantiation for a dtype, vectors per thread, unit size and variant
// (nullptr where U * nv is above kRowsMaxVecs or flags are asked with U > 1).
template <typename T, int MODE>
void* rows_entry_mode(int nv, int unit) {
    switch (nv * 8 + unit) {
        case 1 * 8 + 1: return rows_fn<T, 1, 1, MODE>();
        case 2 * 8 + 1: return rows_fn<T, 2, 1, MODE>();
        case 3 * 8 + 1: return rows_fn<T, 3, 1, MODE>();
        case 4 * 8 + 1: return rows_fn<T, 4, 1, MODE>();
        default: break;
    }
    if constexpr (MODE != kFlags) {
        switch (nv * 8 + unit) {
            case 1 * 8 + 2: return rows_fn<T, 1, 2, MODE>();
            case 1 * 8 + 4: return rows_fn<T, 1, 4, MODE>();
            case 2 * 8 + 2: return rows_fn<T, 2, 2, MODE>();
            default: break;
        }
    }
    return nullptr;
}

template <typename T>
void* rows_entry_for(int nv, int unit, int mode) {
    switch (mode) {
        case kFixed: return rows_entry_mode<T, kFixed>(nv, unit);
        case kClaim: return rows_entry_mode<T, kClaim>(nv, unit);
        case kFlags: return rows_entry_mode<T, kFlags>(nv, unit);
        default: return nullptr;
    }
}

void* rows_kernel_for(int dtype, int nv, int unit, int mode) {
    return dtype == TW_BF16 ? rows_entry_for<__nv_bfloat16>(nv, unit, mode)
                            : rows_entry_for<float>(nv, unit, mode);
}

// y[0..1] = (x[0..1] * inv) * w[0..1], two lanes per instruction (each lane
// rounds as the scalar multiplies do).
__device__ __forceinline__ void scale2(float* y, const float* x, float inv, const float* w) {
    asm("{\n\t.reg .b64 a, b, c;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %4};\n\t"
        "mul.rn.f32x2 a, a, b;\n\t"
        "mov.b64 c, {%5, %6};\n\t"
        "mul.rn.f32x2 a, a, c;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "=f"(y[0]), "=f"(y[1])
        : "f"(x[0]), "f"(x[1]), "f"(inv), "f"(w[0]), "f"(w[1]));
}

// Two pipelines per CTA (fixed schedule only).  The CTA's ring is cut into
// two halves, each with its own producer warp, its own 8 consumer warps and
// its own stages and mbarriers; pipeline g takes the CTA's units at
// positions g, g + 2, g + 4, ... (unit b + i * grid at position i).  Each
// pipeline walks only its own slots in order, so no wait can mistake an
// older phase of a slot for the one it needs.  A consumer group's chain of
// "wait for a stage, read it, release it" then runs beside the other
// group's, and a stage that lands while one group is in its epilogue is
// taken by the other.  Per unit the group meets at its own named barrier
// (ids 1 and 2, 256 threads each).  NV: vectors per consumer thread and row
// with 256 threads per group (U * NV <= kRowsMaxVecs).
template <typename T, int NV, int U>
__global__ void __launch_bounds__(kRowsBlock, 1)
    rows2_kernel(const __grid_constant__ Params p) {
    static_assert(U >= 1 && U <= kRowsMaxUnit && U * NV <= kRowsMaxVecs, "unit too large");
    constexpr int kGroupWarps = kConsumerWarps / 2;
    constexpr int kGroupThreads = kRowsThreads / 2;
    extern __shared__ __align__(1024) unsigned char smem[];
    using V = Vec<T>;
    constexpr int E = V::kElems;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t S = static_cast<uint32_t>(p.stages);  // even: S / 2 per pipeline
    const uint32_t Sg = S / 2;
    const int n_sum = p.colsplit ? 1 : p.n_parts;
    const int R = n_sum + 1;
    const int G = p.rows_per_stage;
    const int stages_per_unit = (R + G - 1) / G;
    const int64_t rb = p.row_bytes;
    const uint32_t group_bytes = static_cast<uint32_t>(U * rb);
    const uint32_t stage_bytes = static_cast<uint32_t>(G) * group_bytes;
    const uint32_t full0 = smem_addr(smem + kFullOff);
    const uint32_t empty0 = smem_addr(smem + kEmptyOff);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
    const unsigned char* ring = smem + kRingOff;
    const uint32_t ring_addr = smem_addr(ring);
    const int64_t n_units = (p.t1 - p.t0 + U - 1) / U;

    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kGroupWarps);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    // L2 warming before the dependency wait, as in rows_kernel.
    if (warp == kConsumerWarps && lane == 0 && p.prefetch) {
        const int64_t unit_bytes = static_cast<int64_t>(R) * U * rb;
        int64_t n_pre = (kPrefetchTokens + U - 1) / U;
        if (n_pre * unit_bytes > kPrefetchMaxBytes) n_pre = kPrefetchMaxBytes / unit_bytes;
        for (int64_t i = 0; i < n_pre; ++i) {
            const int64_t u = blockIdx.x + i * gridDim.x;
            if (u >= n_units) break;
            const int64_t t = p.t0 + u * U;
            const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
            prefetch_tokens(p, t, n_tok, R, n_sum);
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0 && p.smid_log) p.smid_log[blockIdx.x] = sm_id();

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------ producers ---
        const int pw = warp - kConsumerWarps;  // pipeline
        if (lane != 0 || pw >= 2) return;
        const uint64_t pol = policy_evict_first();
        const uint32_t base = static_cast<uint32_t>(pw) * Sg;
        RingPos pos;
        uint64_t issued = 0;
        bool stop = false;
        for (int64_t i = pw; !stop; i += 2) {
            const int64_t u = blockIdx.x + i * gridDim.x;
            if (u >= n_units) break;
            const int64_t t = p.t0 + u * U;
            const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
            const uint32_t copy_bytes = static_cast<uint32_t>(n_tok * rb);
            const int64_t row_off = t * rb;
            for (int k = 0; k < stages_per_unit; ++k, ++issued, pos.advance(Sg)) {
                const uint32_t s = base + pos.stage;
                if (*abort_flag ||
                    (issued >= Sg && !mbar_wait(empty0 + 8 * s, pos.phase ^ 1u, abort_flag))) {
                    give_up(p, abort_flag);
                    stop = true;
                    break;
                }
                const int g0 = k * G;
                const int g1 = g0 + G < R ? g0 + G : R;
                const uint32_t bar = full0 + 8 * s;
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>(g1 - g0) * copy_bytes);
                uint32_t dst = ring_addr + s * stage_bytes;
                for (int g = g0; g < g1; ++g, dst += group_bytes) {
                    if (g == n_sum) {
                        bulk_g2s(dst, static_cast<const char*>(p.residual) + row_off, copy_bytes,
                                 bar, pol);
                    } else if (p.colsplit) {
                        for (int j = 0; j < n_tok; ++j)
                            for (int r = 0; r < p.n_parts; ++r) {
                                const int64_t lo = p.col_lo[r], hi = p.col_lo[r + 1];
                                if (lo < hi)
                                    bulk_g2s(dst + static_cast<uint32_t>(j * rb + lo),
                                             static_cast<const char*>(p.partials[r]) + row_off +
                                                 j * rb + lo,
                                             static_cast<uint32_t>(hi - lo), bar, pol);
                            }
                    } else {
                        bulk_g2s(dst, static_cast<const char*>(p.partials[g]) + row_off,
                                 copy_bytes, bar, pol);
                    }
                }
            }
        }
        // Drain: this pipeline's copies must have landed before the CTA exits.
        RingPos back = pos;
        for (uint32_t k = 0; k < Sg && k < issued; ++k) {
            if (back.stage == 0) {
                back.stage = Sg - 1;
                back.phase ^= 1u;
            } else {
                --back.stage;
            }
            if (!mbar_wait(full0 + 8 * (base + back.stage), back.phase, nullptr))
                atomicOr(p.status, 2u);
        }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int grp = warp / kGroupWarps;
    const int gwarp = warp - grp * kGroupWarps;
    const int gtid = tid - grp * kGroupThreads;
    const uint32_t base = static_cast<uint32_t>(grp) * Sg;
    const int64_t nvec = rb / 16;
    uint4 wv[NV];
#pragma unroll
    for (int jj = 0; jj < NV; ++jj) {
        const int64_t v = static_cast<int64_t>(jj) * kGroupThreads + gtid;
        wv[jj] = v < nvec ? ld_global_nc(static_cast<const char*>(p.weight) + v * 16)
                          : make_uint4(0, 0, 0, 0);
    }
    // Bounded waits; a consumer that gave up keeps walking its group's units
    // (no waits, no stores) so the group's barrier sequence stays whole.
    RingPos pos;
    int red_buf = 0;
    bool alive = true;
    int nv_ok = 0;  // vectors of a row this thread owns
#pragma unroll
    for (int jj = 0; jj < NV; ++jj)
        if (static_cast<int64_t>(jj) * kGroupThreads + gtid < nvec) nv_ok = jj + 1;
    for (int64_t i = grp;; i += 2) {
        const int64_t u = blockIdx.x + i * gridDim.x;
        if (u >= n_units) break;
        const int64_t t = p.t0 + u * U;
        const int n_tok = U == 1 ? 1 : (p.t1 - t < U ? static_cast<int>(p.t1 - t) : U);
        float x[U][NV][E];
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int jj = 0; jj < NV; ++jj)
#pragma unroll
                for (int e = 0; e < E; ++e) x[j][jj][e] = 0.f;
        for (int k = 0; k < stages_per_unit; ++k, pos.advance(Sg)) {
            const uint32_t s = base + pos.stage;
            if (alive && !mbar_wait(full0 + 8 * s, pos.phase, abort_flag)) {
                give_up(p, abort_flag);
                alive = false;
            }
            const int g0 = k * G;
            const int g1 = g0 + G < R ? g0 + G : R;
            const unsigned char* stage = ring + s * stage_bytes + gtid * 16;
            for (int g = g0; g < g1; ++g) {
                const unsigned char* group = stage + (g - g0) * group_bytes;
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    if (U == 1 || j < n_tok) {
                        const unsigned char* row = group + j * rb;
#pragma unroll
                        for (int jj = 0; jj < NV; ++jj)
                            if (jj < nv_ok)
                                add_vec(x[j][jj],
                                        *reinterpret_cast<const uint4*>(
                                            row + jj * kGroupThreads * 16),
                                        static_cast<T*>(nullptr));
                    }
                }
            }
            __syncwarp();
            if (alive && lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // The sum of squares is reduced exactly as rows_kernel reduces it, so
        // both kernels give the same bits: vector jj * 256 + gtid belongs, in
        // rows_kernel, to thread (jj & 1) * 256 + gtid (its vector jj >> 1),
        // i.e. to warp gwarp (even jj) or gwarp + 8 (odd jj).  Each thread
        // keeps the two partials apart, each group warp yields the totals of
        // those two warps, and the 16 totals are added in warp order.
        float* red_unit = red + (grp * 2 + red_buf) * (U * kConsumerWarps);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            float ev2[2] = {0.f, 0.f}, od2[2] = {0.f, 0.f};
#pragma unroll
            for (int jj = 0; jj < NV; ++jj)
                if (static_cast<int64_t>(jj) * kGroupThreads + gtid < nvec) {
                    if ((jj & 1) == 0)
                        sum_squares<E>(ev2, x[j][jj]);
                    else
                        sum_squares<E>(od2, x[j][jj]);
                }
            const float ev = warp_sum(ev2[0] + ev2[1]);
            const float od = warp_sum(od2[0] + od2[1]);
            if (lane == 0) {
                red_unit[j * kConsumerWarps + gwarp] = ev;
                red_unit[j * kConsumerWarps + kGroupWarps + gwarp] = od;
            }
        }
        named_barrier(1 + grp, kGroupThreads);
        red_buf ^= 1;
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (U > 1 && j >= n_tok) break;
            float total = 0.f;
            const float4* r4 = reinterpret_cast<const float4*>(red_unit + j * kConsumerWarps);
#pragma unroll
            for (int w4 = 0; w4 < kConsumerWarps / 4; ++w4) {
                const float4 q4 = r4[w4];
                total += q4.x;
                total += q4.y;
                total += q4.z;
                total += q4.w;
            }
            const float inv = rsqrtf(total * p.inv_H + p.eps);
            const int64_t row_off = (t + j) * rb;
#pragma unroll
            for (int jj = 0; jj < NV; ++jj) {
                const int64_t v = static_cast<int64_t>(jj) * kGroupThreads + gtid;
                if (v < nvec && alive) {
                    st_global_cs(static_cast<char*>(p.residual_out) + row_off + v * 16,
                                 V::from_float(x[j][jj]));
                    float w[E], y[E];
                    V::to_float(wv[jj], w);
#pragma unroll
                    for (int e = 0; e < E; e += 2) scale2(y + e, x[j][jj] + e, inv, w + e);
                    const uint4 packed = V::from_float(y);
                    for (int k = 0; k < p.n_out; ++k)
                        st_global_cs(static_cast<char*>(p.out[k]) + row_off + v * 16, packed);
                }
            }
        }
    }
}

template <typename T>
void* rows2_entry_for(int nv, int unit) {
    switch (nv * 8 + unit) {
        case 1 * 8 + 1: return reinterpret_cast<void*>(&rows2_kernel<T, 1, 1>);
        case 2 * 8 + 1: return reinterpret_cast<void*>(&rows2_kernel<T, 2, 1>);
        case 3 * 8 + 1: return reinterpret_cast<void*>(&rows2_kernel<T, 3, 1>);
        case 4 * 8 + 1: return reinterpret_cast<void*>(&rows2_kernel<T, 4, 1>);
        case 1 * 8 + 2: return reinterpret_cast<void*>(&rows2_kernel<T, 1, 2>);
        case 1 * 8 + 4: return reinterpret_cast<void*>(&rows2_kernel<T, 1, 4>);
        case 2 * 8 + 2: return reinterpret_cast<void*>(&rows2_kernel<T, 2, 2>);
        default: return nullptr;
    }
}

void* rows2_kernel_for(int dtype, int nv, int unit) {
    return dtype == TW_BF16 ? rows2_entry_for<__nv_bfloat16>(nv, unit)
                            : rows2_entry_for<float>(nv, unit);
}

int rows_vectors_per_thread(int64_t row_bytes, int threads = kRowsThreads) {
    return static_cast<int>((row_bytes / 16 + threads - 1) / threads);
}

// Tokens of the busiest CTA when `tokens` tokens are cut into units of u
// (the last one ragged) dealt round robin to min(units, sms) CTAs.
int64_t busiest_cta_tokens(int64_t tokens, int64_t u, int64_t sms) {
    const int64_t units = (tokens + u - 1) / u;
    const int64_t grid = units < sms ? units : sms;
    const int64_t full = (units + grid - 1) / grid;  // units of the busiest CTAs
    const int64_t r = units % grid;
    const int64_t n_busiest = r == 0 ? grid : r;
    if (n_busiest >= 2) return full * u;  // one of them holds whole units only
    // The only busiest CTA (CTA 0) also holds the ragged last unit.
    const int64_t last = tokens - (units - 1) * u;
    return full * u - (u - last);
}

}  // namespace

size_t rows_smem_bytes(size_t stage_bytes, int stages) {
    return static_cast<size_t>(kRingOff) + static_cast<size_t>(stages) * stage_bytes;
}

int rows_unit_tokens(const Params& p, int64_t tokens, int64_t sms) {
    // Units of several tokens only where one copy per row would be small and
    // the unit does not lengthen the busiest CTA's share of the range: the
    // largest U with U * row <= kUnitCopyBytes, U * vectors per thread within
    // the register budget, and the busiest CTA's tokens no more than with
    // one token per unit.  Readiness flags and the column-split mode take
    // one token per unit.
    if (p.ready || p.colsplit || tokens < 1 || sms < 1) return 1;
    const int nv = rows_vectors_per_thread(p.row_bytes);
    const int64_t share1 = busiest_cta_tokens(tokens, 1, sms);
    for (int u = kRowsMaxUnit; u > 1; u /= 2) {
        if (u * p.row_bytes > kUnitCopyBytes || u * nv > kRowsMaxVecs) continue;
        if (busiest_cta_tokens(tokens, u, sms) <= share1) return u;
    }
    return 1;
}

size_t rows_plan(Params& p, int smem_optin) {
    // Whole row groups of one unit per stage: the whole unit if its R groups
    // fit kStageTargetBytes, else the unit's groups split evenly over the
    // fewest stages that fit (never more than R groups).  As many stages as
    // fit the shared memory.  p.unit_tokens must be set.
    const int64_t rows = p.colsplit ? 2 : p.n_parts + 1;
    const int64_t group = p.unit_tokens * p.row_bytes;
    const int64_t parts = (rows * group + kStageTargetBytes - 1) / kStageTargetBytes;
    int64_t per_stage = (rows + parts - 1) / parts;
    if (per_stage * group > kStageTargetBytes) per_stage = kStageTargetBytes / group;
    if (per_stage < 1) per_stage = 1;
    const size_t stage = static_cast<size_t>(per_stage * group);
    int stages = static_cast<int>((static_cast<size_t>(smem_optin) - rows_smem_bytes(0, 0)) / stage);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < kMinStages) return 0;
    // Producer warps: the largest power of two up to kRowsMaxProducers that
    // the ring holds; the ring is cut to a multiple of it, so each producer
    // owns the same stages for the whole launch.
    static_assert((kRowsMaxProducers & (kRowsMaxProducers - 1)) == 0,
                  "producer count must be a power of two");
    int producers = kRowsMaxProducers;
    while (producers > 1 && producers > stages) producers /= 2;
    stages -= stages % producers;
    p.rows_per_stage = static_cast<int>(per_stage);
    p.stages = stages;
    p.producers = producers;
    const size_t smem = rows_smem_bytes(stage, stages);
    return smem < static_cast<size_t>(kExclusiveSmemBytes) ? kExclusiveSmemBytes : smem;
}

bool rows_two_pipes_fit(const Params& p, bool budgeted) {
    // Two pipelines: the fixed schedule, at least two ring stages each, and a
    // unit's x in registers with 256 threads per group.  Under an SM budget
    // they always pay (8 SMs: 291 -> 266 us on N = 8, H = 8192; 190 -> 156
    // us on N = 2, H = 4096).  With the whole GPU only when a pipeline's half
    // of the ring holds a whole unit (N = 2: 14.3 -> 13.6 us); otherwise
    // each pipeline would wait for its own first stage to be read before it
    // could fetch a unit's last one (N = 8: 28.2 -> 28.6 us).
    const int nv2 = rows_vectors_per_thread(p.row_bytes, kRowsThreads / 2);
    if (p.ready || p.work || p.stages < 4 || p.unit_tokens * nv2 > kRowsMaxVecs ||
        rows2_kernel_for(TW_BF16, nv2, p.unit_tokens) == nullptr)
        return false;
    const int rows = p.colsplit ? 2 : p.n_parts + 1;
    const int stages_per_unit = (rows + p.rows_per_stage - 1) / p.rows_per_stage;
    return budgeted || stages_per_unit <= p.stages / 2;
}

int rows_set_smem_limit(int smem_optin) {
    for (int dt = 0; dt < 2; ++dt)
        for (int nv = 1; nv <= kRowsMaxVecs; ++nv)
            for (int unit = 1; unit <= kRowsMaxUnit; unit *= 2)
                for (int mode : {kFixed, kClaim, kFlags}) {
                    void* fn = rows_kernel_for(dt, nv, unit, mode);
                    if (!fn) continue;
                    cudaError_t e = cudaFuncSetAttribute(
                        fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
                    if (e != cudaSuccess) return static_cast<int>(e);
                }
    for (int dt = 0; dt < 2; ++dt)
        for (int nv = 1; nv <= kRowsMaxVecs; ++nv)
            for (int unit = 1; unit <= kRowsMaxUnit; unit *= 2) {
                void* fn = rows2_kernel_for(dt, nv, unit);
                if (!fn) continue;
                cudaError_t e = cudaFuncSetAttribute(
                    fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
                if (e != cudaSuccess) return static_cast<int>(e);
            }
    return 0;
}

int launch_rows(const Params& p, int dtype, int grid, size_t smem_bytes, bool pdl,
                void* stream) {
    void* fn;
    if (p.pipes == 2) {
        fn = rows2_kernel_for(dtype, rows_vectors_per_thread(p.row_bytes, kRowsThreads / 2),
                              p.unit_tokens);
    } else {
        const int mode = p.ready ? kFlags : p.work ? kClaim : kFixed;
        fn = rows_kernel_for(dtype, rows_vectors_per_thread(p.row_bytes), p.unit_tokens, mode);
    }
    if (!fn) return static_cast<int>(cudaErrorInvalidValue);
    return launch_with_pdl(fn, p, grid, kRowsBlock, smem_bytes, pdl, stream);
}

}  // namespace tw
