/*
 * sparse-moe-4bit for GB300 (sm_103a): C ABI of the sparse Mixture-of-Experts
 * block with 4-bit group-affine expert weights.
 *
 * Operation (Perplexity, "Optimizing on-device inference for Apple Silicon",
 * 2026):
 *   - §"Qwen creates three different workload shapes": a router scores E
 *     experts per token and keeps k (256 and 8 in the model the pages study);
 *     one shared expert processes every token.
 *   - §"Dequantize weights during matrix multiplication": each weight is a
 *     4-bit code, each group of 64 weights along K shares a scale s and a
 *     bias beta (value = s*q + beta); the code is expanded tile by tile inside
 *     the matrix multiplication and never written out as a full matrix;
 *     accumulation is fp32.
 *   - §"Keep expert routing on the GPU": histogram, prefix scan, scatter and
 *     block map run on the GPU with no host round-trip inside a layer.
 *   - §"Match tile size to expert load": the tile shape follows each
 *     expert's row count.
 *   - §"Reduce intermediate and state traffic": the output projection is
 *     combined with its routing score and the shared expert's result.
 *   - §"Limiting temporary memory with prompt chunking": long inputs run in
 *     bounded chunks with unchanged output.
 *
 * Per token t (x_t bf16 [d]):
 *   l[e]  = x_t . W_r[e] (+ b_e)                     fp32
 *   top-k experts by (l desc, e asc); w_j = exp(l_j - l_max) / sum over kept
 *   y_e   = D_e (silu(G_e x_t) * (U_e x_t))           SwiGLU, dequantised weights
 *   sigma = sigmoid(w_sg . x_t)
 *   out_t = sum_{j<k} w_j y_{e_j} + sigma * y_shared  (fixed order) -> bf16
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers unless the name ends in _host.
 *     They are caller-owned; the library never frees them.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Every call only enqueues work on that stream (no host
 *     synchronisation inside), except moe_create (one synchronisation at the
 *     end), moe_forward_host (synchronises before returning) and
 *     moe_get_device_error (synchronises the handle's last stream).
 *   - Argument errors are reported before anything is enqueued.  No C++
 *     exception crosses this boundary.  A failed call leaves a message that
 *     moe_last_error() returns (per thread).
 *   - Faults the GPU detects while running (NaN router logits, an internal
 *     wait that ran past its time limit) set a device error word instead of
 *     trapping; read it with moe_get_device_error().
 *   - A handle is not re-entrant: calls on one handle must be ordered (one
 *     stream, or events between streams).
 */
#ifndef SPARSE_MOE_BIT_GB300_MOE_H
#define SPARSE_MOE_BIT_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or config value   */
  MOE_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. group = 96)    */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed                     */
  MOE_ERR_OOM = 4,         /* device allocation failed                       */
  MOE_ERR_DEVICE = 5       /* the device error word is set                   */
} moe_status;

/* Scale/bias storage type of the quantised weights. */
enum { MOE_SCALE_F16 = 1, MOE_SCALE_BF16 = 2 };

/* Which kernel layouts moe_create builds (bitmask; 0 means both).
 * PREFILL serves T > 1 (tensor-core grouped GEMMs), DECODE serves T == 1
 * (bandwidth path) and moe_decode.  Without DECODE, T == 1 runs on the
 * prefill path. */
enum { MOE_LAYOUT_PREFILL = 1, MOE_LAYOUT_DECODE = 2 };

/* Device error word bits (moe_get_device_error). */
enum {
  MOE_DEVERR_WAIT_TIMEOUT = 1,   /* a pipeline wait passed its time limit    */
  MOE_DEVERR_NAN_LOGIT = 2,      /* a router logit was NaN (treated as -inf) */
  MOE_DEVERR_GRID_TIMEOUT = 4,   /* a wait on another CTA passed its limit   */
  MOE_DEVERR_RANGE = 8,          /* a decode router partial sum was outside
                                    +-2^20 (clamped; fixed-point range)     */
  MOE_DEVERR_FP16_RANGE = 16     /* prefill: an fp16 operand overflowed: a
                                    token whose largest activation is above
                                    2^61 times fp16's range (beyond the
                                    per-token scaling), or a non-finite
                                    output (an intermediate silu(gate)*up
                                    beyond fp16's range, for weights far
                                    outside N(0, 0.02), or a non-finite
                                    input); such outputs are not valid      */
};

typedef struct moe_config {
  int d;           /* hidden size; multiple of 256                          */
  int E;           /* routed experts; 1..512                                 */
  int k;           /* experts kept per token; 1..min(E, 16)                  */
  int I;           /* expert intermediate size (routed and shared); mult. 128 */
  int group;       /* quantisation group along K: a multiple of 64 dividing
                      d and I (64 on the pages); else MOE_ERR_UNSUPPORTED    */
  int scale_dtype; /* MOE_SCALE_F16 or MOE_SCALE_BF16 (the pages' format;
                      converted to fp16 at moe_create: exact for 0 and every
                      magnitude in [2^-17, 65504]; a finite value with no
                      exact fp16 value (above 65504, or tiny with bits below
                      2^-24) makes moe_create return MOE_ERR_UNSUPPORTED)   */
  int max_tokens;  /* tokens per internal chunk (workspace is sized for it)  */
  int has_shared;  /* 1: one sigmoid-gated shared expert; 0: none            */
  int layouts;     /* MOE_LAYOUT_* bitmask, 0 = both                         */
} moe_config;

/*
 * Weights in the canonical layout (all DEVICE pointers, read only during
 * moe_create, which makes the handle's own repacked copy; the caller may free
 * them once moe_create returns).
 *   Codes: uint8, two 4-bit codes per byte, the even K index in the low
 *   nibble; matrices are [out][in] row-major, groups contiguous along in.
 *   Scales and biases: 16-bit (scale_dtype), [out][in / group].
 *   gu_*: [E][2I][d/2] codes, [E][2I][d/group] s and beta; rows 0..I-1 are
 *         the gate projection, rows I..2I-1 the up projection.
 *   dn_*: [E][d][I/2] codes, [E][d][I/group] s and beta.
 *   sh_*: the shared expert, same layouts with E = 1 (ignored if !has_shared).
 *   w_router: bf16 [E][d].   w_shared_gate: bf16 [d] (ignored if !has_shared).
 */
typedef struct moe_weights {
  const void* gu_codes;
  const void* gu_scale;
  const void* gu_bias;
  const void* dn_codes;
  const void* dn_scale;
  const void* dn_bias;
  const void* sh_gu_codes;
  const void* sh_gu_scale;
  const void* sh_gu_bias;
  const void* sh_dn_codes;
  const void* sh_dn_scale;
  const void* sh_dn_bias;
  const void* w_router;
  const void* w_shared_gate;
} moe_weights;

typedef struct moe_handle moe_handle;

/* Validate `cfg`, allocate the handle (repacked weights + workspace for
 * cfg->max_tokens tokens) on the current CUDA device, repack `w` on `stream`
 * and synchronise it once.  On success *out owns everything it allocated. */
moe_status moe_create(const moe_config* cfg, const moe_weights* w, void* stream,
                      moe_handle** out);

/* Free everything the handle owns (synchronises the device first). NULL ok. */
moe_status moe_destroy(moe_handle* h);

/*
 * Routing only (router GEMM, softmax/top-k, histogram, scan, scatter), for
 * T <= max_tokens tokens.  x: bf16 [T][d].  logit_bias: fp32 [E] or NULL.
 * Outputs (each may be NULL):
 *   logits_out fp32 [T][E] (bias included), idx int32 [T][k] (slot order:
 *   logit descending, ties to the lower expert), w fp32 [T][k],
 *   counts int32 [E], offsets int32 [E+1], perm int32 [T*k] (token of each
 *   grouped row), slot int32 [T][k] (row of assignment (t, j)).
 */
moe_status moe_route(moe_handle* h, const void* x, int T, const float* logit_bias,
                     float* logits_out, int32_t* idx, float* w, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* slot, void* stream);

/* The same routing outputs from given fp32 logits [T][E] (bias, if any, is
 * added first).  Lets a caller (or a test) route from exactly known logits. */
moe_status moe_route_from_logits(moe_handle* h, const float* logits, int T,
                                 const float* logit_bias, int32_t* idx, float* w,
                                 int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* slot, void* stream);

/*
 * The whole block: y bf16 [T][d] from x bf16 [T][d], any T >= 0 (inputs
 * longer than max_tokens run in chunks of max_tokens; the output does not
 * depend on the chunking).  logit_bias: fp32 [E] or NULL.  x and y must not
 * overlap.  16-byte aligned pointers required.
 */
moe_status moe_forward(moe_handle* h, const void* x, int T, const float* logit_bias,
                       void* y, void* stream);

/* moe_forward on HOST buffers: copies x_host (and bias_host, if not NULL) to
 * the device, runs the block, copies the result to y_host and synchronises
 * `stream` before returning.  Pinned host memory gives asynchronous copies. */
moe_status moe_forward_host(moe_handle* h, const void* x_host, int T,
                            const float* bias_host, void* y_host, void* stream);

/* Optional per-layer outputs of moe_decode (device pointers, each may be NULL). */
typedef struct moe_decode_trace {
  float* logits;   /* fp32 [L][E], the logits the routing used (bias included) */
  int32_t* idx;    /* int32 [L][k] */
  float* w;        /* fp32 [L][k] */
  float* sigma;    /* fp32 [L], shared-expert gate */
  void* out;       /* bf16 [L][d], output of every layer */
  int64_t* timestamps; /* int64 [L][4]: GPU clock (ns) in the first CTA once
                          the layer's router sums and input are complete,
                          after its weight copies are issued, once its
                          partial down projections are written, and once the
                          layer output of its features is summed (profiling
                          aid) */
} moe_decode_trace;

/*
 * Batch-1 decode through L layers (handles built with the DECODE layout and
 * identical d, E, k, I): x_0 = x (bf16 [d]); layer l maps x_l to out_l;
 * x_{l+1} = out_l / sqrt(mean(out_l^2) + eps) (fp32, no learned weight);
 * y (bf16 [d]) = out_{L-1}.  One launch for all L layers.  logit_bias: NULL
 * or fp32 [L][E].
 */
moe_status moe_decode(moe_handle* const* layers, int L, const void* x,
                      const float* logit_bias, float eps, void* y,
                      const moe_decode_trace* trace, void* stream);

/* moe_decode on HOST buffers: copies x_host (bf16 [d]) and bias_host (NULL or
 * fp32 [L][E], L <= 64) to the first layer's staging buffers, runs the chain,
 * copies y to y_host (bf16 [d]) and synchronises `stream`. */
moe_status moe_decode_host(moe_handle* const* layers, int L, const void* x_host,
                           const float* bias_host, float eps, void* y_host, void* stream);

/* Per-stage timing of moe_forward (benchmark aid).  While enabled, every
 * moe_forward call records CUDA events around its stages on the caller's
 * stream: 0 router GEMM, 1 routing (top-k, histogram, scan + tile map,
 * scatter, fp16 copy of the activations + shared gate: one kernel), 2 gate/up
 * GEMM, 3 down GEMM, 4 combine.
 * moe_profile_read synchronises the device, writes the summed milliseconds
 * per stage into ms[0..n-1] (n <= 5) and the
 * number of timed chunks into *calls, and resets the sums.  At most 4096
 * chunks are kept between reads (later ones are not timed). */
moe_status moe_profile_enable(moe_handle* h, int enable);
moe_status moe_profile_read(moe_handle* h, float* ms, int n, int* calls);

/*
 * Routing from given logits (as moe_route_from_logits, no handle, no shared
 * expert) that allocates no device memory.  The pages have no counterpart of
 * this entry point: it exists for callers that cannot call cudaMalloc -- code
 * running inside a device memory allocator or its callbacks, serving loops
 * that must never pay cudaMalloc's implicit device synchronisation, programs
 * whose device memory is entirely owned by another framework.
 *   Scratch: one file-scope device array of about 2.5 MB inside this library,
 *   held by every GPU that loads the library until the process exits.  Limits:
 *   T <= 2048, E <= 256, k <= 16 and k <= E; larger sizes, a NULL output and
 *   a pointer that is not 4-byte aligned return MOE_ERR_INVALID_ARG before
 *   anything is enqueued; a launch that fails returns MOE_ERR_CUDA (errors
 *   of earlier, unrelated launches are neither reported nor cleared).
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the one array: calls that overlap on the GPU (different
 *   streams without ordering) race and give undefined results.
 *   Inputs: logits fp32 [T][E] (device), logit_bias fp32 [E] or NULL.
 *   Outputs (device, all required): idx int32 [T][k], w fp32 [T][k],
 *   counts int32 [E], offsets int32 [E+1], perm int32 [T*k], slot int32 [T][k].
 *   NaN logits are treated as -inf (not reported by this entry point).
 */
moe_status moe_route_from_logits_noalloc(const float* logits, int T, int E, int k,
                                         const float* logit_bias, int32_t* idx, float* w,
                                         int32_t* counts, int32_t* offsets, int32_t* perm,
                                         int32_t* slot, void* stream);

/* Synchronise the stream of the handle's last call and read (then clear) its
 * device error word (MOE_DEVERR_* bits).  Test and debugging aid. */
moe_status moe_get_device_error(moe_handle* h, int* code);

const char* moe_status_string(moe_status s);
const char* moe_last_error(void);
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MOE_BIT_GB300_MOE_H */
