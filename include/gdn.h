/*
 * sparse-moe-4bit for GB300 (sm_103a): C ABI of the Gated DeltaNet prefill
 * scan, exported by the same library as moe.h (libmoe.so) and following its
 * conventions (device pointers, caller-owned buffers, asynchronous on the
 * given stream, argument errors reported before anything is enqueued, the
 * message of a failed call in moe_last_error()).
 *
 * Operation (Perplexity, "Optimizing on-device inference for Apple Silicon",
 * 2026):
 *   - §"Qwen creates three different workload shapes": a Gated DeltaNet
 *     layer folds the tokens before the current one into a recurrent state
 *     of fixed size; a learned gate decides how much of the state is kept,
 *     a delta update writes the current token; every token depends on the
 *     state left by the one before it.
 *   - §"Keep recurrent state on chip": the state is a matrix carried through
 *     the whole prompt in registers and written back once, after the scan;
 *     the state and its gate are fp32, queries and keys bf16.
 *
 * The update, read as the gated delta rule, per value head h and token t of
 * a sequence, in order:
 *   alpha_t = exp(g[t][h])
 *   S_t     = alpha_t S_{t-1} (I - beta[t][h] k_t k_t^T) + beta[t][h] v_t k_t^T
 *   o[t][h] = scale * S_t q_t                                   -> bf16
 * with S [dv][dk] fp32 (it maps keys to values), q_t = q[t][hq], k_t =
 * k[t][hq], v_t = v[t][h] and hq = h / (Hv / Hk) (grouped heads).
 */
#ifndef SPARSE_MOE_BIT_GB300_GDN_H
#define SPARSE_MOE_BIT_GB300_GDN_H

#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Scan N sequences packed one after another along the token axis.
 *
 *   q, k      bf16 [T][Hk][dk], row-major, 16-byte aligned
 *   v         bf16 [T][Hv][dv], 16-byte aligned
 *   g         fp32 [T][Hv], log of the gate (alpha = exp(g); g <= 0 keeps
 *             alpha in (0, 1], which the scan assumes for stability)
 *   beta      fp32 [T][Hv], write strength, normally in [0, 1]
 *   scale     readout scale (1/sqrt(dk) in the usual layer); finite
 *   offsets   int32 [N+1] device array of sequence boundaries (sequence n
 *             is tokens offsets[n] .. offsets[n+1]-1), or NULL for a single
 *             sequence of T tokens (then N must be 1).  Offsets must be
 *             non-decreasing within [0, T]; the kernel clamps each
 *             sequence's range into [0, T] with end >= start, so bad offsets
 *             cannot address memory outside the buffers (ranges that then
 *             overlap write the same rows of o in no defined order).  Tokens
 *             outside every sequence are not written.
 *   state_in  fp32 [N][Hv][dv][dk], 16-byte aligned, or NULL (zero state)
 *   state_out fp32 [N][Hv][dv][dk], 16-byte aligned, or NULL (not written);
 *             may equal state_in (updated in place)
 *   o         bf16 [T][Hv][dv], 16-byte aligned
 *   stream    cudaStream_t as void*; the call only enqueues one kernel
 *
 * q, k, v, g, beta and o may be NULL when T = 0 (then the call only writes
 * state_out: a copy of state_in, or zeros; nothing at all without state_out).
 *
 * Supported: dk = 128; dv a positive multiple of 32; Hv a multiple of Hk;
 * Hv <= 65535 and N <= 65535.  Other dk or dv return MOE_ERR_UNSUPPORTED;
 * NULL required pointers, misalignment, negative sizes or a non-finite scale
 * return MOE_ERR_INVALID_ARG.  Nothing is allocated.
 */
moe_status gdn_scan(const void* q, const void* k, const void* v, const float* g,
                    const float* beta, float scale, const int32_t* offsets, int N, int T,
                    int Hk, int Hv, int dk, int dv, const float* state_in, float* state_out,
                    void* o, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MOE_BIT_GB300_GDN_H */
