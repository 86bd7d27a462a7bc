/*
 * tw_oracle.h -- fp64 CPU oracle for the fused reduce + residual add + RMSNorm
 * hot path of TokenWeave.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this code; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no source, header, helper or
 * constant with the CUDA path.
 *
 * Conventions shared by every entry point:
 *   - All arrays are fp64, row-major [T, H] with row stride H (weight is [H]).
 *     The caller widens bf16/fp32 storage values to fp64 exactly.
 *   - partials is an array of n_parts pointers, one [T, H] tensor per simulated
 *     tensor-parallel rank.  out is an array of n_out pointers, one [T, H]
 *     gather destination per simulated rank.
 *   - Only rows [t0, t1) of residual_out and of every out[k] are written; the
 *     other rows keep whatever the caller put there.
 *   - Return value: 0 on success, -1 on an invalid argument (nothing written).
 */
#ifndef TW_ORACLE_H
#define TW_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Traditional order: AllReduce(sum) over all rows of the range, then every
 * simulated rank k in [0, n_out) runs residual add + RMSNorm on the full
 * reduced tensor and writes its own destination out[k].
 * "TokenWeave 策略详解", §1 背景 (output = RMSNorm(residual + allreduce_output) * weight)
 * and §2 (traditional order AllReduce -> residual add -> RMSNorm). */
int tw_oracle_traditional(const double* const* partials, int n_parts,
                          const double* residual, const double* weight,
                          double* const* out, int n_out, double* residual_out,
                          int64_t T, int64_t H, double eps,
                          int64_t t0, int64_t t1);

/* Reordered order: each of n_parts simulated ranks takes a contiguous token
 * slice of [t0, t1) (ReduceScatter on token boundaries), adds its residual
 * slice, RMS-normalises it, and the AllGather copies every slice into every
 * destination out[k].
 * "TokenWeave 策略详解", §2 (ReduceScatter -> residual add -> RMSNorm -> AllGather)
 * and §3.2-3.4 (token slices per GPU, slice-local residual, gather). */
int tw_oracle_reordered(const double* const* partials, int n_parts,
                        const double* residual, const double* weight,
                        double* const* out, int n_out, double* residual_out,
                        int64_t T, int64_t H, double eps,
                        int64_t t0, int64_t t1);

/* Token slice [*first, *last) of rank r out of n_ranks over n_tokens tokens
 * (relative to the start of the range): floor(r*n/N) .. floor((r+1)*n/N).
 * "TokenWeave 策略详解", §3.2 (tokens split evenly over the GPUs). */
int tw_oracle_token_slice(int64_t n_tokens, int n_ranks, int r,
                          int64_t* first, int64_t* last);

/* Number of threads the oracle's token loops use (1 without OpenMP). */
int tw_oracle_threads(void);

/* Sets the thread count of later calls (n >= 1; other values are ignored).
   Overrides OMP_NUM_THREADS. */
void tw_oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif

#endif /* TW_ORACLE_H */
