// tw_internal.h -- launch parameters shared by the host API and the kernels.
#pragma once

#include <stdint.h>

#include "tw.h"

namespace tw {

// Consumer threads of the rows kernel; thread i owns the 16-byte vectors
// i, i + kRowsThreads, ... of a token row (at most kRowsMaxVecs of them, so a
// row is at most kRowsThreads * kRowsMaxVecs * 16 = 32 KB).
constexpr int kRowsThreads = 512;
constexpr int kRowsMaxVecs = 4;
// Producer warps of the rows kernel (one elected lane each issues the bulk
// copies of the ring stages it owns).  One SM's copy rate grows with the
// number of warps issuing copies, so a CTA that streams alone on its SM
// issues from several.
constexpr int kRowsMaxProducers = 2;
// Target bytes of one ring stage of the rows kernel (whole row groups of one
// unit of tokens, at least one group).
constexpr int kStageTargetBytes = 64 * 1024;
// Tokens per unit of the rows kernel: at most kRowsMaxUnit consecutive tokens,
// so that one bulk copy of a buffer's rows of the unit moves at most
// kUnitCopyBytes (short rows move in larger copies; one issuing warp's copy
// rate grows with the copy size).
constexpr int kRowsMaxUnit = 4;
constexpr int64_t kUnitCopyBytes = 16 * 1024;
// Ring depth bounds of the rows kernel.
constexpr int kMaxStages = 16;
constexpr int kMinStages = 2;
// Dynamic shared memory every rows/warp CTA asks for at least: above half of
// an SM's 228 KB, so no two CTAs of a launch share an SM and a grid of at most
// max_sms CTAs occupies at most max_sms SMs.
constexpr int kExclusiveSmemBytes = 120 * 1024;
// Work counters of the rows kernel per device: a launch that claims units
// dynamically gets a pair of its own, handed out again only once that launch
// has completed (an event per pair).
constexpr int kWorkSlots = 64;
// Warps per CTA of the warp-per-token kernel.
constexpr int kWarpTokensPerCta = 4;
// Cluster kernel: threads per CTA, largest cluster, vectors per thread bound.
constexpr int kClusterThreads = 128;
constexpr int kClusterMaxSize = 16;
constexpr int kClusterMaxVpt = 4;

struct Params {
    const void* partials[TW_MAX_PARTS];
    void* out[TW_MAX_OUTS];
    const void* residual;
    const void* weight;
    void* residual_out;
    uint32_t* smid_log;     // optional, rows kernel only
    unsigned int* status;   // device status word (bounded-wait give-ups)
    // Rows kernel: this launch's work counter pair (next unit to claim, CTAs
    // done claiming), zero at launch; NULL: a fixed unit schedule.
    unsigned int* work;
    int64_t t0, t1;         // token range
    int64_t row_bytes;      // H * element size (multiple of 16)
    int64_t H;
    // Column-split mode (rows kernel): partial r is zero outside the byte
    // range [col_lo[r], col_lo[r + 1]) of each row, which alone is read; the
    // staged chunk then holds the concatenation in one row.
    int64_t col_lo[TW_MAX_PARTS + 1];
    // Readiness flags (rows kernel): when `ready` is not NULL, token t is read
    // only once ready[t / block_tokens] has reached `epoch` (wrap-safe).
    const unsigned int* ready;
    int64_t block_tokens;
    unsigned int epoch;
    int n_parts, n_out;
    int unit_tokens;        // rows kernel: consecutive tokens per unit (1, 2 or 4)
    int pipes;              // rows kernel: 1, or 2 independent pipelines per CTA
    int rows_per_stage;     // rows kernel: row groups (one buffer's rows of a unit) per stage
    int stages;             // rows kernel: ring depth (a multiple of producers)
    int producers;          // rows kernel: producer warps issuing copies (1..kRowsMaxProducers)
    int colsplit;           // 1: column-split mode
    int prefetch;           // 1: warm L2 before the dependency wait (overlapped launches)
    float eps;
    float inv_H;
};

// Record `message` as the calling thread's last error and return `code`.
int set_last_error(int code, const char* message);

// Launchers (return a cudaError_t value as int).  `pdl` launches with
// programmatic stream serialization: the kernel may start while the previous
// kernel of the stream drains, and waits (griddepcontrol.wait) before its
// first global memory access.
int launch_rows(const Params& p, int dtype, int grid, size_t smem_bytes, bool pdl,
                void* stream);
// Shared memory the warp kernel needs to keep every warp's token x between
// its two passes (above the device's opt-in limit: the two-pass kernel).
size_t warp_stage_bytes(int64_t row_bytes, int dtype);
int launch_warp(const Params& p, int dtype, int grid, size_t smem_bytes, bool staged, bool pdl,
                void* stream);
// Shared memory of the rows kernel for a stage size and ring depth.
size_t rows_smem_bytes(size_t stage_bytes, int stages);
// Tokens per unit of the rows kernel for a range of `tokens` tokens on at
// most `sms` CTAs (p's row_bytes, ready and colsplit set).
int rows_unit_tokens(const Params& p, int64_t tokens, int64_t sms);
// Launch plan of the rows kernel for p (row_bytes, n_parts, colsplit and
// unit_tokens set): sets rows_per_stage, stages and producers and returns the
// dynamic shared memory to request, or 0 if the rows do not fit in
// smem_optin bytes.
size_t rows_plan(Params& p, int smem_optin);
// Whether the launch planned in p (fixed schedule, unit size and ring set)
// runs as two pipelines per CTA (`budgeted`: held below the SM count).
bool rows_two_pipes_fit(const Params& p, bool budgeted);
// Raise the dynamic shared memory limit of every kernel instantiation on the
// current device (cudaError_t as int).
int rows_set_smem_limit(int smem_optin);
int warp_set_smem_limit(int smem_optin);
int cluster_set_attributes(int smem_optin);
// Load the readiness-flag producer kernel (tw_set_ready) on the current
// device (cudaError_t as int).
int signal_prepare();
// Vectors per thread the cluster kernel needs (0: the row is too long).
int cluster_vectors_per_thread(int64_t row_bytes, int cluster);
// Clusters of `cluster` CTAs of the cluster kernel instantiation for dtype,
// vpt vectors per thread and np partials held in registers (2, 4, 8 or 16),
// each CTA with smem_bytes of dynamic shared memory, that the current device
// can run at once (cudaError_t as int).
int cluster_max_active(int cluster, size_t smem_bytes, int dtype, int vpt, int np, int* n);
// Partials the cluster kernel holds in registers for n_parts partials.
int cluster_np(int n_parts);
int launch_cluster(const Params& p, int dtype, int cluster, int n_clusters, size_t smem_bytes,
                   bool pdl, void* stream);

}  // namespace tw
