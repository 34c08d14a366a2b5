// Batch-1 decode path: one persistent cooperative kernel runs every layer of
// the chain on CUDA cores.  The work is bound by weight reads (4.5 bits per
// weight): each CTA streams only its share of the selected experts' weights
// into shared memory with bulk (TMA) copies issued as soon as the routing is
// known, and computes while they land.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Optimizing the one-row weight path" (a row-parallel GEMV: a SIMD group
// cooperates on one output while reading different parts of the weight
// matrix), §"Reduce intermediate and state traffic" (gate and up projections
// fused with their gated activation; the output projection fused with its
// routing score and the shared expert's result) and §"Keep each decode step
// on the GPU" (no host synchronisation between steps).
//
// The k+1 active experts' intermediate features are cut into blocks of 32
// (one expert each); CTA c takes blocks c, c+G, ... and, for a block, computes
// its 32 gated features h = silu(G x) * (U x) and at once their share of the
// output projection, w_j * D_j[:, block] h_block, over all d output features
// (the "partial" of the block).  So h never leaves the CTA; only the partials
// are exchanged.  CTA c also owns the output features [c*d/G, (c+1)*d/G).
//
// There is no grid-wide barrier: every value one CTA hands to another carries
// the proof of its own completeness in the same machine word, and the reader
// polls the data itself (one L2 round trip after the last writer, where a
// barrier followed by a read costs two):
//   * a partial is a 64-bit word (fp32 value, 32-bit tag of launch and
//     layer), stored and loaded as one single-copy-atomic access;
//   * an output feature is a 32-bit word (bf16 value, 16-bit layer tag);
//   * the router sums are 64-bit fixed-point integers (2^-32 units) added
//     with atomics into one of several copies, each addend also adding 1 to
//     an arrival count in the top 6 bits; a copy is complete when its count
//     equals the number of CTAs that add into it.  Integer addition makes the
//     sum exact and independent of the order of arrival.
// One layer:
//   A : poll the router sums P_l and the previous output out_{l-1}; fold
//       1/rms(out_{l-1}) into the logits (the rest of the layer works on the
//       unnormalised vector and scales its dot products); top-k over the
//       whole CTA (rank within 32-expert chunks, then among the chunks'
//       candidates); bulk copies of the block's gate/up rows (one per warp)
//       and down columns.
//   B : gate/up of the block (two features per warp), h of the block to
//       16-bit integers, the block's tagged partial over all d outputs.
//   C : poll the partials of the owned features, out[f] = their sum in a
//       fixed order, rounded to bf16 and published; the next layer's router
//       sums over the owned features, P_{l+1}[e] += sum_f out[f] W_r'[e][f].
// A CTA whose block belongs to the shared expert (known without routing)
// issues the next layer's copies as soon as its buffers are free.
// Dot products use the split s*q + beta per 64-group:
//   sum_i (s q_i + beta) x_i = s sum_i q_i x_i + beta X,   X = sum_i x_i,
// with sum_i q_i x_i an exact integer dot product (dp2a: two 16-bit inputs
// times two 4-bit codes per instruction) of the codes and the inputs held as
// 16-bit integers with one power-of-two scale per group of inputs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "ptx.cuh"
#include "softmax_df.cuh"
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kBlk = 32;                        // intermediate features per block
constexpr int kUnitsPerWarp = kBlk / kDecWarps;  // gate/up features a warp computes
static_assert(kUnitsPerWarp == 2, "gate/up takes two features per warp");
constexpr int kMaxDecLayers = 64;
constexpr int kPCopies = 8;  // copies of the router sums: CTA c adds into copy c % kPCopies
constexpr int kCountShift = 58;                      // arrival count: bits 58..63
constexpr long long kPOffset = 1ll << 52;            // added to every addend (keeps it >= 0)
constexpr long long kPMaxAbs = (1ll << 52) - 1;      // |addend| limit (2^20 in value)
constexpr int kMaxPerCopy = 31;                      // 31 * 2^53 < 2^58: no carry into the count
constexpr int kRedChunks = 32;  // partial sums per owned feature in the reduction
constexpr int kPollMax = 8;     // partials in flight per thread in one polling pass
constexpr int kMaxOwned = 16;   // owned output features summed per pass (router sums)
constexpr uint64_t kDrainNs = 100000000ull;
// A wait looks at the abort flag (another CTA gave up) only once it has run
// this long: the flag is a global load, one loaded L2 round trip (1-2 us while
// the weights stream), which a wait that reads it at its first retry adds to
// every exchange and copy it waits for.
constexpr uint64_t kAbortCheckNs = 20000ull;

struct DecLayer {
  const uint8_t* gu;     // [n_exp][I] units of d + d/8 bytes (gate, up codes; their s,b)
  const uint8_t* dnc;    // [n_exp][I/32][d] 16 bytes: the 32 codes of a block in row f
  const uint32_t* dnsb;  // [n_exp][I/64][d] scale/bias word of row f, input group g
  const uint16_t* w_rt;  // [d][Ep] router transposed + shared-gate column
};

struct DecParams {
  DecLayer layer[kMaxDecLayers];
  int L, d, E, k, I, has_shared, Ep;
  int nf_max;  // output features per CTA (max)
  int NB;      // blocks per layer: (k+1 or k) * I / 32
  unsigned epoch;  // launch number: part of the partials' tags
  const uint16_t* x;
  int norm_first;  // 1: x is an earlier layer's output (normalise it first)
  const float* bias;  // [L][E] or null
  float eps;
  uint16_t* y;
  float* logits;        // [L][E]
  float* sigma;         // [L]
  int32_t* tr_idx;      // [L][k] or null
  float* tr_w;          // [L][k] or null
  uint16_t* tr_out;     // [L][d] or null
  int64_t* tr_ns;       // [L][4] or null
  unsigned long long* part;  // [NB][d] tagged partial outputs of the blocks
  uint32_t* out;        // [2][d] tagged outputs: layer l writes row l % 2; zero at launch
  unsigned long long* P;  // [L][kPCopies][E+1] counted fixed-point router sums, zero at launch
  int* abort_flag;      // zero at launch
  int* err;
  uint64_t wait_ns;     // a wait on another CTA or a copy gives up after this
  // test of the give-up path: wait for one more router-sum arrival than any
  // CTA makes (a flag that nothing sets); the wait must run out
  int unset_flag;
};

// shared-memory carve-up (the host sizes the launch with the same function)
struct DecSmem {
  size_t xq, xsc, xg, xraw, gu, dnc, dnsb, hb, hpk, rt, outs, red2, lg, lb, keys, cand, sel_e, sel_w,
      misc, red, infl, bars, total;
};
__host__ __device__ inline size_t dec_take(size_t& o, size_t bytes, size_t align) {
  o = (o + align - 1) / align * align;
  const size_t r = o;
  o += bytes;
  return r;
}
__host__ __device__ inline DecSmem dec_smem(int d, int E, int Ep, int nf_max) {
  DecSmem s;
  size_t o = 0;
  const int nch = (E + 31) / 32;
  s.xq = dec_take(o, (size_t)d * 2, 16);
  s.xsc = dec_take(o, (size_t)(d / 64) * 4, 16);
  s.xg = dec_take(o, (size_t)(d / 64) * 4, 16);
  s.xraw = dec_take(o, (size_t)d * 2, 16);
  s.gu = dec_take(o, (size_t)kBlk * (d + d / 8), 128);
  s.dnc = dec_take(o, (size_t)d * 16, 128);
  s.dnsb = dec_take(o, (size_t)d * 4, 128);
  s.hb = dec_take(o, (size_t)kBlk * 4, 16);
  s.hpk = dec_take(o, (size_t)(kBlk / 8) * 16, 16);
  s.rt = dec_take(o, (size_t)nf_max * Ep * 2, 128);
  s.outs = dec_take(o, (size_t)nf_max * 4, 16);
  s.red2 = dec_take(o, (size_t)kRedChunks * 16 * 4, 16);
  s.lg = dec_take(o, (size_t)(E + 1) * 4, 16);
  s.lb = dec_take(o, (size_t)E * 4, 16);
  s.keys = dec_take(o, (size_t)max(nch, 8) * 32 * 8, 16);   // >= 256 keys (small top-k)
  s.cand = dec_take(o, (size_t)nch * kMaxK * 8, 16);
  s.sel_e = dec_take(o, kMaxK * 4, 16);
  s.sel_w = dec_take(o, kMaxK * 4, 16);
  s.misc = dec_take(o, 16, 16);
  s.red = dec_take(o, kDecWarps * 4, 16);
  s.infl = dec_take(o, (kDecWarps + 2) * 4, 16);
  s.bars = dec_take(o, (kDecWarps + 2) * 8, 8);
  s.total = o;
  return s;
}

__device__ __forceinline__ float bf16f(uint32_t v) { return __uint_as_float(v << 16); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float s_of(uint32_t sb) {
  return __half2float(__ushort_as_half((uint16_t)(sb & 0xFFFFu)));
}
__device__ __forceinline__ float b_of(uint32_t sb) {
  return __half2float(__ushort_as_half((uint16_t)(sb >> 16)));
}


// d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (.lo) or bytes 2, 3 (.hi);
// a signed 16-bit pairs, b unsigned bytes
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Activations enter the dot products as 16-bit integers with one power-of-two
// scale 2^e per group of 64, e = floor(log2 amax) - 13 so that every value of
// the group is below 2^14 units: a bf16 value within 2^6 of its group's
// maximum is represented exactly, any other value to within 2^-15 of the
// group maximum.  This holds over fp32's whole range: amax below 2^-99
// (subnormal included) is scaled by 2^64 before its exponent is read, and
// e >= -149 keeps the scale 2^e representable.
__device__ __forceinline__ int group_exponent(float amax) {
  int ex;  // floor(log2 amax)
  if (amax < 1.0e-30f)
    ex = (int)((__float_as_uint(amax * 18446744073709551616.0f) >> 23) & 0xFFu) - 127 - 64;
  else
    ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  return max(ex - 13, -149);
}
// 2^-e for a group exponent e >= -126 (a normal float)
__device__ __forceinline__ float inv_pow2(int e) { return __int_as_float((127 - e) << 23); }
// 2^e, exact also where it is subnormal (two power-of-two factors)
__device__ __forceinline__ float pow2(int e) {
  const int a = e >> 1, b = e - a;
  return __int_as_float((a + 127) << 23) * __int_as_float((b + 127) << 23);
}
// fp32 bits whose low 16 bits are round(v * 2^-e) as a 16-bit integer:
// adding 1.5 * 2^23 leaves the rounded integer in the low mantissa bits.
// Below e = -126, 2^-e exceeds fp32's range: v is first scaled by 2^64
// (exact: such groups are below 2^-99).
__device__ __forceinline__ uint32_t quant_bits(float v, int e) {
  if (e >= -126) return __float_as_uint(fmaf(v, inv_pow2(e), 12582912.0f));
  return __float_as_uint(fmaf(v * 18446744073709551616.0f, inv_pow2(e + 64), 12582912.0f));
}
// the low 16 bits of lo and of hi as one signed 16-bit pair
__device__ __forceinline__ uint32_t pack_lo16(uint32_t lo, uint32_t hi) {
  return __byte_perm(lo, hi, 0x5410);
}
// sum over the 8 codes of word w (K indices 8m..8m+7, two per byte, low
// nibble first) of q * v, with v packed as (v0,v2), (v4,v6), (v1,v3), (v5,v7)
__device__ __forceinline__ int dot8i(uint32_t w, uint4 v, int acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // q0 q2 q4 q6
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // q1 q3 q5 q7
  acc = dp2a_lo(v.x, lo, acc);
  acc = dp2a_hi(v.y, lo, acc);
  acc = dp2a_lo(v.z, hi, acc);
  return dp2a_hi(v.w, hi, acc);
}


// Single-copy-atomic accesses of another CTA's data at GPU scope (the L1
// cache is not used, so a poll sees the latest value in L2).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a));
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* a, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
// four 32-bit words, each read atomically on its own
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* a) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(a));
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* a, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_u64(unsigned long long* a, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

// Pacing of a poll on another CTA's data (each round is one L2 round trip;
// no sleep: a sleeping poller measured up to ~2 us late); gives up (true)
// when another CTA gave up (looked at after kAbortCheckNs) or, recording the
// error, after p.wait_ns.
template <class PP>
__device__ __forceinline__ bool poll_give_up(const PP& p, uint64_t& t0, uint32_t& n) {
  ++n;
  if ((n & 15u) == 1u) {
    const uint64_t t = globaltimer_ns();
    if (n == 1u) {
      t0 = t;
    } else if (t - t0 > kAbortCheckNs) {
      if (*(volatile int*)p.abort_flag) return true;
      if (t - t0 > p.wait_ns) {
        atomicOr(p.err, MOE_DEVERR_GRID_TIMEOUT);
        atomicExch(p.abort_flag, 1);
        return true;
      }
    }
  }
  return false;
}

// Top-k of T tokens over the whole CTA, ranked by (value descending, index
// ascending).  keys[t][e] (e < 32 * chunks) = order key of expert e's logit
// << 32 | ~e, 0 past E: distinct, larger is better; cand[] zero; both
// written by the caller before a barrier.  An expert's rank within its chunk
// of 32 makes the chunk's k best candidates (an expert of the overall top k
// has fewer than k better experts anywhere, so also in its chunk); a
// candidate's rank among its token's candidates is then its overall rank:
// sel_e[t * kMaxK + rank] for rank < k.  Two threads count for a key (16
// comparisons each), and 512 / (all candidates) threads, a power of two, for
// a candidate.
__device__ __forceinline__ void cta_topk(const unsigned long long* keys, unsigned long long* cand,
                                         int E, int k, int T, int* sel_e, int tid) {
  const int nch = (E + 31) >> 5, nkey = 32 * nch, nc = nch * k;
  // whole warps in every pass (the shuffles); keys past E are 0
  for (int it = tid; it < T * 64 * nch; it += kDecThreads) {
    const int tok = it / (64 * nch), r = it - tok * 64 * nch;
    const int e = r >> 1, h = r & 1;
    const unsigned long long* kt = keys + tok * nkey;
    const unsigned long long my = kt[e];
    const unsigned long long* kc = kt + (e & ~31) + 16 * h;
    int rank = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) rank += (kc[i] > my) ? 1 : 0;
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    if (h == 0 && e < E && rank < k) cand[tok * nc + (e >> 5) * k + rank] = my;
  }
  __syncthreads();
  int tpc = 32;  // threads per candidate
  while (tpc > 1 && tpc * nc * T > kDecThreads) tpc >>= 1;
  const int tot = (T * nc * tpc + 31) & ~31;
  for (int it = tid; it < tot; it += kDecThreads) {
    const int ci = it / tpc, part = it % tpc;  // candidate over all tokens
    const bool ok = ci < T * nc;
    const int tok = ok ? ci / nc : 0;
    const unsigned long long* ct = cand + tok * nc;
    const unsigned long long my = ok ? ct[ci - tok * nc] : 0ull;
    int rank = 0;
    if (ok)
      for (int j = part; j < nc; j += tpc) rank += (ct[j] > my) ? 1 : 0;
    for (int o = 1; o < tpc; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (part == 0 && my != 0ull && rank < k)
      sel_e[tok * kMaxK + rank] = (int)(0xFFFFFFFFu - (uint32_t)my);
  }
  __syncthreads();
}

// round(v * 2^32) as a 64-bit integer for |v| < 2^20, from 32-bit
// conversions (the 64-bit ones are slow): x = v 2^32 is exact; its high part
// floor(x / 2^24) and the remainder x - hi 2^24 (in [0, 2^24), exact) convert
// exactly, the remainder rounded to nearest even.
__device__ __forceinline__ long long fix32(float v) {
  const float x = v * 4294967296.0f;
  const float hi = floorf(x * 5.9604644775390625e-8f);  // 2^-24
  const float rem = fmaf(-hi, 16777216.0f, x);
  return (long long)__float2int_rn(hi) * 16777216ll + (long long)__float2int_rn(rem);
}
// a 64-bit integer s (|s| < 2^62) times 2^-32 in fp32: the sum of its two
// 32-bit halves, each converted exactly or within half an ulp
__device__ __forceinline__ float unfix32(long long s) {
  const int hi = (int)(s >> 32);
  const unsigned lo = (unsigned)(s & 0xFFFFFFFFll);
  return fmaf((float)lo, 2.3283064365386963e-10f, (float)hi);  // lo 2^-32 + hi
}

// Bounded wait on an mbarrier phase; the thread sleeps in hardware between
// checks.  On time-out (or when another CTA gave up) records the error.
template <class PP>
__device__ __forceinline__ bool copy_wait(const PP& p, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const uint64_t t = globaltimer_ns();
    if (t - t0 < kAbortCheckNs) continue;
    if (*(volatile int*)p.abort_flag) return false;
    if (t - t0 > p.wait_ns) {
      atomicOr(p.err, MOE_DEVERR_WAIT_TIMEOUT);
      atomicExch(p.abort_flag, 1);
      return false;
    }
  }
}

// Four consecutive activations v0..v3 at index i0 (a multiple of 4; the 16
// lanes of a half-warp hold one group of 64) -> 16-bit integers with the
// group's power-of-two scale, stored as the packed pairs the integer dot
// products take: word m of group g holds (x0,x2), (x4,x6), (x1,x3),
// (x5,x7) of K indices 8m..8m+7.  Also the group's scale and sum.  Every
// lane of the warp takes part (shuffles); act = false contributes nothing.
__device__ __forceinline__ void quant_x4_into(float v0, float v1, float v2, float v3, int i0,
                                              bool act, uint4* xq, float* xsc, float* xg, int ng,
                                              int lane) {
  float am = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
  float sum = (v0 + v1) + (v2 + v3);
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
  }
  const int e = group_exponent(am);
  const uint32_t b0 = quant_bits(v0, e), b1 = quant_bits(v1, e);
  const uint32_t b2 = quant_bits(v2, e), b3 = quant_bits(v3, e);
  if (act) {
    const int g = i0 >> 6, kk = i0 & 63;
    uint32_t* wp = reinterpret_cast<uint32_t*>(xq + (kk >> 3) * ng + g);
    const int h4 = (kk & 4) ? 1 : 0;  // second half of the word: x4..x7
    wp[h4] = pack_lo16(b0, b2);
    wp[2 + h4] = pack_lo16(b1, b3);
    if ((lane & 15) == 0) {
      xsc[g] = pow2(e);
      xg[g] = sum;
    }
  }
}

// One warp's share of a block's gate/up: the warp's two features (units u =
// 0, 1 at ub0, gu_unit bytes each: gate codes, up codes, gate s,b, up s,b),
// for each token t < NTOK in tmask (its activations at xq + t * xstride, its
// group scales and sums at xsc, xg + t * sstride); lane: one group of 64
// inputs at a time, the group's code words loaded once for every token.
// acc[t] = the lane's partial sums (gate u0, up u0, gate u1, up u1); the
// caller sums the warp.  sum_i (s q_i + beta) x_i = s sum_i q_i x_i + beta X
// per group (X = sum_i x_i); the same expressions for every NTOK, so a
// token's sums do not depend on the other tokens.
template <int NTOK>
__device__ __forceinline__ void gateup_rows(const uint8_t* ub0, int gu_unit, int d, int ng,
                                            const uint4* xq, const float* xsc, const float* xg,
                                            int xstride, int sstride, unsigned tmask, int lane,
                                            float (&acc)[NTOK][4]) {
#pragma unroll
  for (int t = 0; t < NTOK; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  for (int g = lane; g < ng; g += 32) {
    uint4 cw[2][4];
    uint32_t sbg[2], sbu[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint8_t* ub = ub0 + u * gu_unit;
      cw[u][0] = *reinterpret_cast<const uint4*>(ub + g * 32);
      cw[u][1] = *reinterpret_cast<const uint4*>(ub + g * 32 + 16);
      cw[u][2] = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32);
      cw[u][3] = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32 + 16);
      sbg[u] = reinterpret_cast<const uint32_t*>(ub + d)[g];
      sbu[u] = reinterpret_cast<const uint32_t*>(ub + d + d / 16)[g];
    }
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      if (!((tmask >> t) & 1u)) continue;
      const uint4* xt = xq + t * xstride;
      uint4 xw[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) xw[m] = xt[m * ng + g];
      const float sc = xsc[t * sstride + g], X = xg[t * sstride + g];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint4 cg0 = cw[u][0], cg1 = cw[u][1], cu0 = cw[u][2], cu1 = cw[u][3];
        int pg0 = dot8i(cg0.x, xw[0], 0), pg1 = dot8i(cg0.y, xw[1], 0);
        int pu0 = dot8i(cu0.x, xw[0], 0), pu1 = dot8i(cu0.y, xw[1], 0);
        pg0 = dot8i(cg0.z, xw[2], pg0);
        pg1 = dot8i(cg0.w, xw[3], pg1);
        pu0 = dot8i(cu0.z, xw[2], pu0);
        pu1 = dot8i(cu0.w, xw[3], pu1);
        pg0 = dot8i(cg1.x, xw[4], pg0);
        pg1 = dot8i(cg1.y, xw[5], pg1);
        pu0 = dot8i(cu1.x, xw[4], pu0);
        pu1 = dot8i(cu1.y, xw[5], pu1);
        pg0 = dot8i(cg1.z, xw[6], pg0);
        pg1 = dot8i(cg1.w, xw[7], pg1);
        pu0 = dot8i(cu1.z, xw[6], pu0);
        pu1 = dot8i(cu1.w, xw[7], pu1);
        acc[t][2 * u] += s_of(sbg[u]) * (sc * (float)(pg0 + pg1)) + b_of(sbg[u]) * X;
        acc[t][2 * u + 1] += s_of(sbu[u]) * (sc * (float)(pu0 + pu1)) + b_of(sbu[u]) * X;
      }
    }
  }
}

// h of a 32-feature block (lane = feature, one warp) -> 16-bit integers with
// one power-of-two scale, packed as the integer dot products take them
// (word m: features 8m..8m+7); also the scale and the sum of h.  qt: 32 words
// of scratch.
__device__ __forceinline__ void quant_h32(float v, uint32_t* qt, uint4* hpk, float* hsc, float* hs,
                                          int lane) {
  float am = fabsf(v), s = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  const int e = group_exponent(am);
  qt[lane] = quant_bits(v, e);
  __syncwarp();
  if (lane < kBlk / 8) {
    const uint32_t* q8 = qt + lane * 8;
    hpk[lane] = make_uint4(pack_lo16(q8[0], q8[2]), pack_lo16(q8[4], q8[6]),
                           pack_lo16(q8[1], q8[3]), pack_lo16(q8[5], q8[7]));
  }
  if (lane == 0) {
    *hsc = pow2(e);
    *hs = s;
  }
}

// One output row's share of a block's down projection, times the routing
// weight wj: wj (s sum_i q_i h_i + beta H) over the block's 32 features
// (cw: their codes in row f; sb: the row's scale/bias word of the block's
// input group; h packed as quant_h32 leaves it).
__device__ __forceinline__ float down_value(uint4 cw, uint32_t sb, uint4 h0, uint4 h1, uint4 h2,
                                            uint4 h3, float hsc, float Hs, float wj) {
  const int a = (dot8i(cw.x, h0, 0) + dot8i(cw.y, h1, 0)) + (dot8i(cw.z, h2, 0) + dot8i(cw.w, h3, 0));
  return wj * (s_of(sb) * (hsc * (float)a) + b_of(sb) * Hs);
}

__device__ __forceinline__ void stamp(const DecParams& p, int l, int i) {
  if (p.tr_ns && blockIdx.x == 0 && threadIdx.x == 0)
    p.tr_ns[(long long)l * 4 + i] = (int64_t)globaltimer_ns();
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int d = p.d, E = p.E, k = p.k, I = p.I, Ep = p.Ep;
  const int ng = d / 64;
  const int NB = p.NB;
  const int bpe = I / kBlk;  // blocks per expert
  const int nch = (E + 31) >> 5;
  const DecSmem L = dec_smem(d, E, Ep, p.nf_max);
  uint4* xq = reinterpret_cast<uint4*>(dsm + L.xq);   // [8 words][ng] packed int16 x
  float* xsc = reinterpret_cast<float*>(dsm + L.xsc);  // [ng] scale of a group of x
  float* xg = reinterpret_cast<float*>(dsm + L.xg);    // [ng] sum of a group of x
  uint16_t* xraw = reinterpret_cast<uint16_t*>(dsm + L.xraw);  // [d] previous output, bf16
  uint8_t* gu_buf = dsm + L.gu;                        // [32 units] of d + d/8 bytes
  const uint4* dnc = reinterpret_cast<const uint4*>(dsm + L.dnc);        // [d] block codes
  const uint32_t* dnsb = reinterpret_cast<const uint32_t*>(dsm + L.dnsb);  // [d] s,b words
  float* hb = reinterpret_cast<float*>(dsm + L.hb);    // [32] h of the block
  uint4* hpk = reinterpret_cast<uint4*>(dsm + L.hpk);  // [4 words] packed int16 h
  const uint16_t* rt_buf = reinterpret_cast<const uint16_t*>(dsm + L.rt);
  float* outs = reinterpret_cast<float*>(dsm + L.outs);
  float* red2 = reinterpret_cast<float*>(dsm + L.red2);  // [chunks][16] reduction partials
  float* lg = reinterpret_cast<float*>(dsm + L.lg);      // logits
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(dsm + L.keys);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(dsm + L.cand);
  int* sel_e = reinterpret_cast<int*>(dsm + L.sel_e);
  float* sel_w = reinterpret_cast<float*>(dsm + L.sel_w);
  float* misc = reinterpret_cast<float*>(dsm + L.misc);  // [0] sigma [1] 1/rms [2] h scale [3] h sum
  float* red = reinterpret_cast<float*>(dsm + L.red);
  // parity of the copies in flight on each mbarrier (-1: none), for the
  // bounded drain on the error path
  volatile int* infl = reinterpret_cast<volatile int*>(dsm + L.infl);
  const uint32_t bar0 = smem_u32(dsm + L.bars);  // [warps] gate/up, then down, router
  const int kDnBar = kDecWarps, kRtBar = kDecWarps + 1;
  const uint32_t dn_bar = bar0 + 8 * kDnBar;
  const uint32_t rt_bar = bar0 + 8 * kRtBar;
  const int wwarp = kDecWarps - 1;  // computes the routing weights
  // bulk copies other than a warp's own gate/up rows (the issuing thread
  // waits for each): down columns by warp 14, router rows by warp 15
  constexpr int kDnTid = (kDecWarps - 2) * 32 + 1, kRtTid = (kDecWarps - 1) * 32 + 31;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int f0 = (int)((long long)c * d / G), f1 = (int)((long long)(c + 1) * d / G);
  const int nf = f1 - f0;
  const int gu_unit = d + d / 8;

  if (tid == 0) {
    for (int i = 0; i < kDecWarps + 2; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (tid < kDecWarps + 2) infl[tid] = -1;
  __syncthreads();
  uint32_t ph_gu = 0, ph_dn = 0, ph_rt = 0;
  bool pre = false;  // the CTA's first block of this layer was issued during the last one

  // Error path: wait, with a bound, for this CTA's bulk copies still in
  // flight, so that none lands in shared memory after the CTA has left.
  auto drain = [&]() {
    if (lane != 0) return;
    for (int i = 0; i < kDecWarps + 2; ++i) {
      const int pty = infl[i];
      if (pty < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar0 + 8 * i, (uint32_t)pty)) {
        if (globaltimer_ns() - t0 > kDrainNs) break;
      }
    }
  };

  // Block b: expert slot j = b / bpe (slot k: the shared expert), features
  // (b % bpe) * 32 .. + 31.  issue_gu (lane 0 of each warp): the gate/up rows
  // of the warp's two features; issue_dn (one thread): the block's down
  // columns (codes of every output row, then the rows' scale/bias words of
  // its input group).
  auto issue_gu = [&](int b, const DecLayer& W) {
    const int j = b / bpe, i0 = (b - j * bpe) * kBlk;
    const long long ex = (j < k) ? sel_e[j] : E;
    const uint32_t bar = bar0 + 8 * warp;
    const uint32_t bytes = (uint32_t)(kUnitsPerWarp * gu_unit);
    infl[warp] = (int)ph_gu;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(gu_buf + (size_t)warp * kUnitsPerWarp * gu_unit),
             W.gu + (ex * I + i0 + warp * kUnitsPerWarp) * gu_unit, bytes, bar);
  };
  auto issue_dn = [&](int b, const DecLayer& W) {
    const int j = b / bpe, i0 = (b - j * bpe) * kBlk;
    const long long ex = (j < k) ? sel_e[j] : E;
    infl[kDnBar] = (int)ph_dn;
    mbar_arrive_expect_tx(dn_bar, (uint32_t)(d * 20));
    bulk_g2s(smem_u32(dsm + L.dnc), W.dnc + (ex * bpe + i0 / kBlk) * (long long)d * 16,
             (uint32_t)(d * 16), dn_bar);
    bulk_g2s(smem_u32(dsm + L.dnsb), W.dnsb + (ex * (I / 64) + i0 / 64) * (long long)d,
             (uint32_t)(d * 4), dn_bar);
  };

  auto quant_x4 = [&](float v0, float v1, float v2, float v3, int i0, bool act) {
    quant_x4_into(v0, v1, v2, v3, i0, act, xq, xsc, xg, ng, lane);
  };

  // x (bf16 [d]) -> quantised activations in shared memory, with optional
  // RMS normalisation; also the owned features' values (used for the input
  // of the first layer of a launch).
  auto load_x = [&](const uint16_t* src, bool norm) {
    float r = 1.0f;
    if (norm) {
      float ss = 0.f;
      for (int i = tid; i < d; i += kDecThreads) {
        const float v = bf16f(__ldg(src + i));
        ss += v * v;
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < kDecWarps; ++w) t += red[w];
        misc[1] = rsqrtf(t / (float)d + p.eps);
      }
      __syncthreads();
      r = misc[1];
    }
    for (int ib = 0; ib < d; ib += 4 * kDecThreads) {
      const int i0 = ib + 4 * tid;
      const bool act = i0 < d;
      uint2 raw = make_uint2(0u, 0u);
      if (act) raw = __ldg(reinterpret_cast<const uint2*>(src + i0));
      const float v[4] = {bf16f(raw.x & 0xFFFFu) * r, bf16f(raw.x >> 16) * r,
                          bf16f(raw.y & 0xFFFFu) * r, bf16f(raw.y >> 16) * r};
      quant_x4(v[0], v[1], v[2], v[3], i0, act);
      if (act) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i0 + q >= f0 && i0 + q < f1) outs[i0 + q - f0] = v[q];
      }
    }
    __syncthreads();
  };

  // Router sums of layer ln over the owned features, added into copy
  // c % kPCopies of P_ln with one arrival each: P[e] += 2^58 + 2^52 +
  // round(2^32 sum_{f owned} outs[f] W'[e][f]) (e = E: the shared gate).
  // Every CTA adds to every entry (zero without owned features), so that the
  // counts reach their known totals.
  auto router_partial = [&](int ln) {
    unsigned long long* Pq =
        p.P + ((long long)ln * kPCopies + (c % kPCopies)) * (long long)(E + 1);
    bool range_err = false;
    for (int e = tid; e <= E; e += kDecThreads) {
      // every load of the entry first (nf <= kMaxOwned), then the sum
      float acc = 0.f;
      for (int f0 = 0; f0 < nf; f0 += kMaxOwned) {
        uint16_t wv[kMaxOwned];
        float ov[kMaxOwned];
#pragma unroll
        for (int i = 0; i < kMaxOwned; ++i) {
          wv[i] = (f0 + i < nf) ? rt_buf[(f0 + i) * Ep + e] : (uint16_t)0;
          ov[i] = (f0 + i < nf) ? outs[f0 + i] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kMaxOwned; ++i) acc = fmaf(ov[i], bf16f(wv[i]), acc);
      }
      long long v;
      if (fabsf(acc) < 1048575.0f) {
        v = fix32(acc);
      } else {  // outside the fixed-point range (or NaN): clamped, error bit
        v = (acc > 0.0f) ? kPMaxAbs : -kPMaxAbs;
        range_err = true;
      }
      red_add_u64(Pq + e, (1ull << kCountShift) + (unsigned long long)(v + kPOffset));
    }
    if (range_err) atomicOr(p.err, MOE_DEVERR_RANGE);
  };

  // The router sum of entry e of P_ln, once every copy's count is complete.
  // With `ow` (not null), the four tagged output words at `osrc` are polled
  // in the same loop until each carries the tag `otag`: the previous layer's
  // outputs are published before its router sums, so both are ready
  // together and one round trip serves both.
  auto poll_P = [&](const unsigned long long* Ps, int e, long long& sum,
                    const uint32_t* osrc = nullptr, uint32_t otag = 0u,
                    uint4* ow = nullptr) -> bool {
    unsigned long long w[kPCopies];
#pragma unroll
    for (int q = 0; q < kPCopies; ++q) w[q] = ld_relaxed_u64(Ps + q * (E + 1) + e);
    if (ow) *ow = ld_relaxed_v4(osrc);
    uint64_t t0 = 0;
    uint32_t n = 0;
    for (;;) {
      unsigned pend = 0;
#pragma unroll
      for (int q = 0; q < kPCopies; ++q) {
        const unsigned want = ((G > q) ? (unsigned)((G - q + kPCopies - 1) / kPCopies) : 0u) +
                              ((q == 0 && p.unset_flag) ? 1u : 0u);
        if ((unsigned)(w[q] >> kCountShift) != want) pend |= 1u << q;
      }
      const bool opend = ow && ((ow->x >> 16) != otag || (ow->y >> 16) != otag ||
                                (ow->z >> 16) != otag || (ow->w >> 16) != otag);
      if (!pend && !opend) break;
      if (poll_give_up(p, t0, n)) return false;
#pragma unroll
      for (int q = 0; q < kPCopies; ++q)
        if ((pend >> q) & 1u) w[q] = ld_relaxed_u64(Ps + q * (E + 1) + e);
      if (opend) *ow = ld_relaxed_v4(osrc);
    }
    sum = 0;
#pragma unroll
    for (int q = 0; q < kPCopies; ++q) {
      const long long cnt = (long long)(w[q] >> kCountShift);
      sum += (long long)(w[q] & ((1ull << kCountShift) - 1ull)) - cnt * kPOffset;
    }
    return true;
  };

  auto issue_router_copy = [&](int l) {
    if (tid == kRtTid && nf > 0) {
      const uint32_t bytes = (uint32_t)nf * Ep * 2;
      infl[kRtBar] = (int)ph_rt;
      mbar_arrive_expect_tx(rt_bar, bytes);
      bulk_g2s(smem_u32(dsm + L.rt), p.layer[l].w_rt + (long long)f0 * Ep, bytes, rt_bar);
    }
  };

  // ---- prologue: x_0 and the router sums of layer 0
  issue_router_copy(0);
  load_x(p.x, p.norm_first != 0);
  if (nf > 0) {
    if (!copy_wait(p, rt_bar, ph_rt)) {
      drain();
      return;
    }
    if (tid == kRtTid) infl[kRtBar] = -1;
  }
  ph_rt ^= 1;
  router_partial(0);

  for (int l = 0; l < p.L; ++l) {
    const DecLayer& W = p.layer[l];
    const uint32_t ptag = ((p.epoch << 6) | (uint32_t)l) | 0x80000000u;  // partials of layer l
    // ---- A: the router sums P_l (entry e = tid, and E when E = kDecThreads)
    //      and the previous output, polled in one pass
    bool bad = false;
    const unsigned long long* Ps = p.P + (long long)l * kPCopies * (E + 1);
    const uint32_t* osrc = p.out + (long long)((l - 1) & 1) * d;
    const uint32_t otag = (uint32_t)l;  // tag of layer l-1's outputs
    // this thread's first four output words ride along with its P entry
    const bool o_first = l > 0 && tid <= E && 4 * tid < d;
    uint4 oraw = make_uint4(0u, 0u, 0u, 0u);
    long long ps0 = 0, ps1 = 0;
    if (tid <= E && !poll_P(Ps, tid, ps0, osrc + 4 * tid, otag, o_first ? &oraw : nullptr))
      bad = true;
    if (tid + kDecThreads <= E && !poll_P(Ps, tid + kDecThreads, ps1)) bad = true;
    if (l > 0) {
      const uint32_t* src = osrc;
      const uint32_t want = otag;
      float ss = 0.f;
      for (int ib = 0; ib < d; ib += 4 * kDecThreads) {
        const int i0 = ib + 4 * tid;
        const bool act = i0 < d;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (act && !bad) {
          raw = (ib == 0 && o_first) ? oraw : ld_relaxed_v4(src + i0);
          uint64_t t0 = 0;
          uint32_t n = 0;
          while ((raw.x >> 16) != want || (raw.y >> 16) != want || (raw.z >> 16) != want ||
                 (raw.w >> 16) != want) {
            if (poll_give_up(p, t0, n)) {
              bad = true;
              break;
            }
            raw = ld_relaxed_v4(src + i0);
          }
        }
        const float v0 = bf16f(raw.x & 0xFFFFu), v1 = bf16f(raw.y & 0xFFFFu);
        const float v2 = bf16f(raw.z & 0xFFFFu), v3 = bf16f(raw.w & 0xFFFFu);
        ss = fmaf(v0, v0, ss);
        ss = fmaf(v1, v1, ss);
        ss = fmaf(v2, v2, ss);
        ss = fmaf(v3, v3, ss);
        // quantised after the copies are issued (off the routing's path)
        if (act)
          *reinterpret_cast<uint2*>(xraw + i0) =
              make_uint2(pack_lo16(raw.x, raw.y), pack_lo16(raw.z, raw.w));
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
    }
    if (__syncthreads_or(bad)) {
      drain();
      return;
    }
    stamp(p, l, 0);
    float r = 1.0f;  // 1/rms of out_{l-1} (x_0 is normalised already)
    if (l > 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) t += red[w];
      r = rsqrtf(t / (float)d + p.eps);
    }
    // logits, the shared gate, and the top-k keys
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = tid + i * kDecThreads;
      if (e > E) continue;
      float v = unfix32(i == 0 ? ps0 : ps1) * r;
      if (e < E) {
        if (p.bias) v += __ldg(p.bias + (long long)l * E + e);
        lg[e] = v;
        if (c == 0) p.logits[(long long)l * E + e] = v;
        if (v != v) {
          v = -INFINITY;
          nan_seen = true;
        }
        keys[e] = ((unsigned long long)ord_key(v) << 32) |
                  (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
      } else {
        const float sg = p.has_shared ? 1.0f / (1.0f + expf(-v)) : 0.0f;
        misc[0] = sg;
        if (c == 0) p.sigma[l] = sg;
      }
    }
    for (int e = E + tid; e < max(nch, 8) * 32; e += kDecThreads) keys[e] = 0ull;
    if (E > 256)
      for (int i = tid; i < nch * k; i += kDecThreads) cand[i] = 0ull;
    if (__syncthreads_or(nan_seen) && c == 0 && tid == 0) atomicOr(p.err, MOE_DEVERR_NAN_LOGIT);
    if (E <= 256) {  // one warp: lane l takes experts 8l .. 8l+7
      if (warp == 0) {
        unsigned long long s8[8];
        const ulonglong2* kp = reinterpret_cast<const ulonglong2*>(keys + 8 * lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const ulonglong2 q = kp[i];
          s8[2 * i] = q.x;
          s8[2 * i + 1] = q.y;
        }
        const unsigned long long kw = warp_topk_lists(s8, k, lane);
        if (lane < k) sel_e[lane] = (int)(0xFFFFFFFFu - (uint32_t)kw);
      }
      __syncthreads();
    } else {
      cta_topk(keys, cand, E, k, 1, sel_e, tid);
    }
    if (c < NB && !pre) {
      if (lane == 0) issue_gu(c, W);
      if (tid == kDnTid) issue_dn(c, W);
    }
    pre = false;
    stamp(p, l, 1);
    if (l > 0) {  // the previous output -> quantised activations
      for (int ib = 0; ib < d; ib += 4 * kDecThreads) {  // whole warps (shuffles)
        const int i0 = ib + 4 * tid;
        const bool act = i0 < d;
        uint2 raw = make_uint2(0u, 0u);
        if (act) raw = *reinterpret_cast<const uint2*>(xraw + i0);
        quant_x4(bf16f(raw.x & 0xFFFFu), bf16f(raw.x >> 16), bf16f(raw.y & 0xFFFFu),
                 bf16f(raw.y >> 16), i0, act);
      }
      __syncthreads();
    }
    if (warp == wwarp) {
      // routing weights (softmax over the k chosen logits in double-float
      // arithmetic, within one ulp of fp64), off the path of the copies and
      // of the other warps' gate/up work
      const int my_e = (lane < k) ? sel_e[lane] : 0;
      float my_v = (lane < k) ? lg[my_e] : -INFINITY;
      if (my_v != my_v) my_v = -INFINITY;
      float top = lg[sel_e[0]];
      if (top != top) top = -INFINITY;
      const dflt ex = (lane < k) ? df_softmax_term(my_v, top) : dflt{0.0f, 0.0f};
      dflt den = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const dflt ot = {__shfl_xor_sync(0xffffffffu, den.hi, o),
                         __shfl_xor_sync(0xffffffffu, den.lo, o)};
        den = df_add(den, ot);
      }
      if (lane < k) {
        const float wv = df_div(ex, den).hi;
        sel_w[lane] = wv;
        if (c == 0) {
          if (p.tr_idx) p.tr_idx[(long long)l * k + lane] = my_e;
          if (p.tr_w) p.tr_w[(long long)l * k + lane] = wv;
        }
      }
      // the next layer's router rows (read at the end of this layer; the
      // buffer's last reads were before this layer's first barrier)
      if (l + 1 < p.L) issue_router_copy(l + 1);
    }

    // ---- B: the CTA's blocks: gate/up, h, and the block's tagged partial
    for (int b = c, nb = 0; b < NB; b += G, ++nb) {
      const int j = b / bpe;
      if (nb > 0) {
        __syncthreads();  // the previous block's buffers are no longer read
        if (lane == 0) issue_gu(b, W);
        if (tid == kDnTid) issue_dn(b, W);
      }
      // gate/up: warp -> features 2*warp, 2*warp + 1 of the block; lane: one
      // group of 64 inputs at a time, its activations in registers for both
      if (!copy_wait(p, bar0 + 8 * warp, ph_gu)) {
        drain();
        return;
      }
      if (lane == 0) infl[warp] = -1;
      ph_gu ^= 1;
      {
        const uint8_t* ub0 = gu_buf + (size_t)warp * kUnitsPerWarp * gu_unit;
        float acc[1][4];
        gateup_rows<1>(ub0, gu_unit, d, ng, xq, xsc, xg, 0, 0, 1u, lane, acc);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float gv = warp_sum(acc[0][2 * t]) * r, uv = warp_sum(acc[0][2 * t + 1]) * r;
          if (lane == 0) hb[warp * kUnitsPerWarp + t] = gv / (1.0f + expf(-gv)) * uv;
        }
      }
      __syncthreads();
      // h of the block -> 16-bit integers with one power-of-two scale, packed
      // as the integer dot products take them (word m: features 8m..8m+7)
      if (warp == 0)
        quant_h32(hb[lane], reinterpret_cast<uint32_t*>(red2), hpk, &misc[2], &misc[3], lane);
      if (!copy_wait(p, dn_bar, ph_dn)) {
        drain();
        return;
      }
      if (tid == kDnTid) infl[kDnBar] = -1;
      ph_dn ^= 1;
      __syncthreads();
      // the block's partial output: part[b][f] = w_j (s sum_i q_i h_i + beta H),
      // published with the layer's tag
      {
        const uint4 h0 = hpk[0], h1 = hpk[1], h2 = hpk[2], h3 = hpk[3];
        const float hsc = misc[2], Hs = misc[3];
        const float wj = (j < k) ? sel_w[j] : misc[0];
        unsigned long long* pb = p.part + (long long)b * d;
        const unsigned long long tg = (unsigned long long)ptag << 32;
        for (int f = tid; f < d; f += kDecThreads) {
          const float v = down_value(dnc[f], dnsb[f], h0, h1, h2, h3, hsc, Hs, wj);
          st_relaxed_u64(pb + f, tg | __float_as_uint(v));
        }
      }
    }
    // The next layer's first block of this CTA belongs to the shared expert:
    // its weights do not depend on the routing, so they load now.
    if (l + 1 < p.L && p.has_shared && c < NB && c / bpe == k) {
      __syncthreads();  // this layer's buffers are no longer read
      if (lane == 0) issue_gu(c, p.layer[l + 1]);
      if (tid == kDnTid) issue_dn(c, p.layer[l + 1]);
      pre = true;
    }
    stamp(p, l, 2);

    // ---- C: out[f] = sum over blocks of part[b][f] (fixed order), bf16,
    //      published with the layer's tag
    {
      uint32_t* outl = p.out + (long long)(l & 1) * d;
      const uint32_t otag = (uint32_t)(l + 1) << 16;
      for (int fl0 = 0; fl0 < nf; fl0 += 16) {
        const int fl = fl0 + (tid & 15), ch = tid >> 4;  // 32 chunks of blocks
        float s = 0.f;
        if (fl < nf) {
          const unsigned long long* pf = p.part + f0 + fl;
          for (int bp = ch; bp < NB && !bad; bp += kRedChunks * kPollMax) {
            unsigned long long v[kPollMax];
#pragma unroll
            for (int i = 0; i < kPollMax; ++i) {
              const int b = bp + i * kRedChunks;
              v[i] = (b < NB) ? ld_relaxed_u64(pf + (long long)b * d)
                              : ((unsigned long long)ptag << 32);
            }
            uint64_t t0 = 0;
            uint32_t n = 0;
            for (;;) {
              unsigned pend = 0;
#pragma unroll
              for (int i = 0; i < kPollMax; ++i)
                if ((uint32_t)(v[i] >> 32) != ptag) pend |= 1u << i;
              if (!pend) break;
              if (poll_give_up(p, t0, n)) {
                bad = true;
                break;
              }
#pragma unroll
              for (int i = 0; i < kPollMax; ++i)
                if ((pend >> i) & 1u) v[i] = ld_relaxed_u64(pf + (long long)(bp + i * kRedChunks) * d);
            }
#pragma unroll
            for (int i = 0; i < kPollMax; ++i)
              if (bp + i * kRedChunks < NB) s += __uint_as_float((uint32_t)v[i]);
          }
        }
        red2[ch * 16 + (tid & 15)] = s;
        if (__syncthreads_or(bad)) {
          drain();
          return;
        }
        if (tid < 16 && fl0 + tid < nf) {
          float o = 0.f;
          for (int q = 0; q < kRedChunks; ++q) o += red2[q * 16 + tid];
          const uint16_t ob = __bfloat16_as_ushort(__float2bfloat16_rn(o));
          const int f = f0 + fl0 + tid;
          outs[fl0 + tid] = bf16f(ob);
          st_relaxed_u32(outl + f, otag | ob);
          if (p.tr_out) p.tr_out[(long long)l * d + f] = ob;
          if (l == p.L - 1) p.y[f] = ob;
        }
        __syncthreads();
      }
    }
    stamp(p, l, 3);
    if (l + 1 < p.L) {
      if (nf > 0) {
        if (!copy_wait(p, rt_bar, ph_rt)) {
          drain();
          return;
        }
        if (tid == kRtTid) infl[kRtBar] = -1;
      }
      ph_rt ^= 1;
      router_partial(l + 1);
    }
  }
}

// ---------------------------------------------------------------------------
// A few tokens (2 <= T <= kFewMax) of one layer in one launch: every token is
// routed on the device, the union of the experts the tokens picked is formed,
// and each block of an expert in that union is streamed once, for every token
// that picked it (the speculative-verify shape: a handful of rows that pick
// different experts, where one pass of the one-row path per token reads the
// shared experts' weights T times and the matrix path pays whole-tile costs).
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Limits of further optimization" (verify passes of 2-5 rows that pick
// different experts fall between the one-row weight path and the matrix
// path) and §"Optimizing the one-row weight path".
//
// Per token the arithmetic is the decode kernel's (router sums as counted
// 64-bit fixed point over the owned features, the same top-k and softmax, the
// same integer dot products, the same fixed-order sum of the partials), so a
// token's output does not depend on the other tokens of the launch: T copies
// of one token give the decode kernel's single-layer output, bit for bit.
//
// Union entry u = 0 is the shared expert (when there is one), then the routed
// experts in ascending index.  Block b: entry b / bpe, features (b % bpe) *
// 32 .. + 31; CTA c takes blocks c, c + G, ...  The shared expert's blocks do
// not depend on the routing, so CTAs c < bpe issue their first copies at the
// start.  A block computes h for each token that picked its expert and that
// token's partial over all d outputs, tagged, at part[t][slot][b % bpe][f]; a
// warp's gate/up rows of the CTA's next block load as soon as the warp has
// used its current ones, the next down columns once the current ones are
// used.  CTA c owns output features [c d / G, (c+1) d / G) of every token.
constexpr int kFewMax = 8;
constexpr int kFewUnion = kFewMax * kMaxK + 1;  // union entries at most
constexpr int kFewPairs = 2;  // (token, entry) router sums polled together per thread

struct FewParams {
  DecLayer W;
  int T, d, E, k, I, has_shared, Ep, nf_max;
  unsigned epoch;
  const uint16_t* x;         // bf16 [T][d]
  const float* bias;         // [E] or null
  uint16_t* y;               // bf16 [T][d]
  float* logits;             // [T][E] (written by CTA 0)
  unsigned long long* part;  // [T][k1][bpe][d] tagged partials
  unsigned long long* P;     // [T][kPCopies][E+1] counted router sums, zero at launch
  int* abort_flag;           // zero at launch
  int* err;
  uint64_t wait_ns;          // a wait on another CTA or a copy gives up after this
};

struct FewSmem {
  size_t xq, xsc, xg, gu, dnc, dnsb, rt, outs, lg, keys, cand, sel_e, sel_w, sig, umask, ubase,
      ulist, uslot, hb, hpk, hsc, hsum, qt, red2, misc, infl, bars, total;
};
__host__ __device__ inline FewSmem few_smem(int T, int d, int E, int Ep, int nf_max) {
  FewSmem s;
  size_t o = 0;
  s.xq = dec_take(o, (size_t)T * d * 2, 16);
  s.xsc = dec_take(o, (size_t)T * (d / 64) * 4, 16);
  s.xg = dec_take(o, (size_t)T * (d / 64) * 4, 16);
  s.gu = dec_take(o, (size_t)kBlk * (d + d / 8), 128);
  s.dnc = dec_take(o, (size_t)d * 16, 128);
  s.dnsb = dec_take(o, (size_t)d * 4, 128);
  s.rt = dec_take(o, (size_t)nf_max * Ep * 2, 128);
  s.outs = dec_take(o, (size_t)T * nf_max * 4, 16);
  s.lg = dec_take(o, (size_t)T * (E + 1) * 4, 16);
  s.keys = dec_take(o, (size_t)T * ((E + 31) / 32) * 32 * 8, 16);
  s.cand = dec_take(o, (size_t)T * ((E + 31) / 32) * kMaxK * 8, 16);
  s.sel_e = dec_take(o, (size_t)T * kMaxK * 4, 16);
  s.sel_w = dec_take(o, (size_t)T * kMaxK * 4, 16);
  s.sig = dec_take(o, (size_t)T * 4, 16);
  s.umask = dec_take(o, (size_t)(kMaxE / 32) * 4, 16);
  s.ubase = dec_take(o, (size_t)(kMaxE / 32) * 4, 16);
  s.ulist = dec_take(o, (size_t)kFewUnion * 4, 16);
  s.uslot = dec_take(o, (size_t)kFewUnion * kFewMax, 16);
  s.hb = dec_take(o, (size_t)T * kBlk * 4, 16);
  s.hpk = dec_take(o, (size_t)T * (kBlk / 8) * 16, 16);
  s.hsc = dec_take(o, (size_t)T * 4, 16);
  s.hsum = dec_take(o, (size_t)T * 4, 16);
  s.qt = dec_take(o, (size_t)kFewMax * kBlk * 4, 16);
  s.red2 = dec_take(o, (size_t)2 * kRedChunks * 16 * 4, 16);
  s.misc = dec_take(o, 16, 16);
  s.infl = dec_take(o, (kDecWarps + 2) * 4, 16);
  s.bars = dec_take(o, (kDecWarps + 2) * 8, 8);
  s.total = o;
  return s;
}

__global__ void __launch_bounds__(kDecThreads, 1) few_kernel(const __grid_constant__ FewParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int T = p.T, d = p.d, E = p.E, k = p.k, I = p.I, Ep = p.Ep;
  const int ng = d / 64;
  const int bpe = I / kBlk;
  const int k1 = k + (p.has_shared ? 1 : 0);
  const FewSmem L = few_smem(T, d, E, Ep, p.nf_max);
  uint4* xq = reinterpret_cast<uint4*>(dsm + L.xq);    // [T][8 words][ng] packed int16 x
  float* xsc = reinterpret_cast<float*>(dsm + L.xsc);  // [T][ng]
  float* xg = reinterpret_cast<float*>(dsm + L.xg);    // [T][ng]
  uint8_t* gu_buf = dsm + L.gu;
  const uint4* dnc = reinterpret_cast<const uint4*>(dsm + L.dnc);
  const uint32_t* dnsb = reinterpret_cast<const uint32_t*>(dsm + L.dnsb);
  const uint16_t* rt_buf = reinterpret_cast<const uint16_t*>(dsm + L.rt);
  float* outs = reinterpret_cast<float*>(dsm + L.outs);  // [T][nf_max] owned input values
  float* lg = reinterpret_cast<float*>(dsm + L.lg);      // [T][E+1]; entry E: shared gate
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(dsm + L.keys);  // [T][nch*32]
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(dsm + L.cand);  // [T][nch*k]
  int* sel_e = reinterpret_cast<int*>(dsm + L.sel_e);    // [T][kMaxK]
  float* sel_w = reinterpret_cast<float*>(dsm + L.sel_w);
  float* sig = reinterpret_cast<float*>(dsm + L.sig);    // [T]
  uint32_t* umask = reinterpret_cast<uint32_t*>(dsm + L.umask);
  int* ubase = reinterpret_cast<int*>(dsm + L.ubase);
  int* ulist = reinterpret_cast<int*>(dsm + L.ulist);    // union entry -> expert
  int8_t* uslot = reinterpret_cast<int8_t*>(dsm + L.uslot);  // [entry][kFewMax] slot, -1 none
  float* hb = reinterpret_cast<float*>(dsm + L.hb);      // [T][32]
  uint4* hpk = reinterpret_cast<uint4*>(dsm + L.hpk);    // [T][4]
  float* hsc = reinterpret_cast<float*>(dsm + L.hsc);
  float* hsum = reinterpret_cast<float*>(dsm + L.hsum);
  uint32_t* qt = reinterpret_cast<uint32_t*>(dsm + L.qt);  // [kFewMax][32]
  float* red2 = reinterpret_cast<float*>(dsm + L.red2);
  int* misc = reinterpret_cast<int*>(dsm + L.misc);      // [0] union entries
  volatile int* infl = reinterpret_cast<volatile int*>(dsm + L.infl);
  const uint32_t bar0 = smem_u32(dsm + L.bars);
  const int kDnBar = kDecWarps, kRtBar = kDecWarps + 1;
  const uint32_t dn_bar = bar0 + 8 * kDnBar;
  const uint32_t rt_bar = bar0 + 8 * kRtBar;
  constexpr int kDnTid = (kDecWarps - 2) * 32 + 1, kRtTid = (kDecWarps - 1) * 32 + 31;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int f0 = (int)((long long)c * d / G), f1 = (int)((long long)(c + 1) * d / G);
  const int nf = f1 - f0;
  const int gu_unit = d + d / 8;
  const DecLayer& W = p.W;

  if (tid == 0) {
    for (int i = 0; i < kDecWarps + 2; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (tid < kDecWarps + 2) infl[tid] = -1;
  __syncthreads();
  uint32_t ph_gu = 0, ph_dn = 0;

  auto drain = [&]() {
    if (lane != 0) return;
    for (int i = 0; i < kDecWarps + 2; ++i) {
      const int pty = infl[i];
      if (pty < 0) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar0 + 8 * i, (uint32_t)pty)) {
        if (globaltimer_ns() - t0 > kDrainNs) break;
      }
    }
  };
  // copies of block b of expert ex: the warp's gate/up rows (lane 0 of each
  // warp), the block's down columns and their scale/bias words (one thread)
  auto issue_gu = [&](int b, long long ex) {
    const int i0 = (b % bpe) * kBlk;
    const uint32_t bar = bar0 + 8 * warp;
    const uint32_t bytes = (uint32_t)(kUnitsPerWarp * gu_unit);
    infl[warp] = (int)ph_gu;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(gu_buf + (size_t)warp * kUnitsPerWarp * gu_unit),
             W.gu + (ex * I + i0 + warp * kUnitsPerWarp) * gu_unit, bytes, bar);
  };
  auto issue_dn = [&](int b, long long ex) {
    const int i0 = (b % bpe) * kBlk;
    infl[kDnBar] = (int)ph_dn;
    mbar_arrive_expect_tx(dn_bar, (uint32_t)(d * 20));
    bulk_g2s(smem_u32(dsm + L.dnc), W.dnc + (ex * bpe + i0 / kBlk) * (long long)d * 16,
             (uint32_t)(d * 16), dn_bar);
    bulk_g2s(smem_u32(dsm + L.dnsb), W.dnsb + (ex * (I / 64) + i0 / 64) * (long long)d,
             (uint32_t)(d * 4), dn_bar);
  };

  // ---- the shared expert's first block (no routing needed) and the router
  //      rows of the owned features
  const bool pre = p.has_shared && c < bpe;
  if (pre) {
    if (lane == 0) issue_gu(c, E);
    if (tid == kDnTid) issue_dn(c, E);
  }
  if (tid == kRtTid && nf > 0) {
    const uint32_t bytes = (uint32_t)nf * Ep * 2;
    infl[kRtBar] = 0;
    mbar_arrive_expect_tx(rt_bar, bytes);
    bulk_g2s(smem_u32(dsm + L.rt), W.w_rt + (long long)f0 * Ep, bytes, rt_bar);
  }

  // ---- every token's activations -> quantised, and the owned features'
  //      values (the loads of all tokens first)
  for (int ib = 0; ib < d; ib += 4 * kDecThreads) {
    const int i0 = ib + 4 * tid;
    const bool act = i0 < d;
    uint2 rawt[kFewMax];
#pragma unroll
    for (int t = 0; t < kFewMax; ++t)
      rawt[t] = (act && t < T) ? __ldg(reinterpret_cast<const uint2*>(p.x + (long long)t * d + i0))
                               : make_uint2(0u, 0u);
#pragma unroll
    for (int t = 0; t < kFewMax; ++t) {
      if (t >= T) break;
      const uint2 raw = rawt[t];
      const float v[4] = {bf16f(raw.x & 0xFFFFu), bf16f(raw.x >> 16), bf16f(raw.y & 0xFFFFu),
                          bf16f(raw.y >> 16)};
      quant_x4_into(v[0], v[1], v[2], v[3], i0, act, xq + (size_t)t * 8 * ng, xsc + t * ng,
                    xg + t * ng, ng, lane);
      if (act) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i0 + q >= f0 && i0 + q < f1) outs[t * p.nf_max + i0 + q - f0] = v[q];
      }
    }
  }
  __syncthreads();

  // ---- router sums of every token over the owned features (CTA c adds into
  //      copy c % kPCopies of each entry, zero without owned features)
  if (nf > 0) {
    if (!copy_wait(p, rt_bar, 0)) {
      drain();
      return;
    }
    if (tid == kRtTid) infl[kRtBar] = -1;
  }
  {
    bool range_err = false;
    for (int e = tid; e <= E; e += kDecThreads) {
      for (int t = 0; t < T; ++t) {
        // the decode kernel's order: owned features in chunks of kMaxOwned
        const float* ot = outs + t * p.nf_max;
        float acc = 0.f;
        for (int fb = 0; fb < nf; fb += kMaxOwned) {
          uint16_t wv[kMaxOwned];
          float ov[kMaxOwned];
#pragma unroll
          for (int i = 0; i < kMaxOwned; ++i) {
            wv[i] = (fb + i < nf) ? rt_buf[(fb + i) * Ep + e] : (uint16_t)0;
            ov[i] = (fb + i < nf) ? ot[fb + i] : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < kMaxOwned; ++i) acc = fmaf(ov[i], bf16f(wv[i]), acc);
        }
        long long v;
        if (fabsf(acc) < 1048575.0f) {
          v = fix32(acc);
        } else {
          v = (acc > 0.0f) ? kPMaxAbs : -kPMaxAbs;
          range_err = true;
        }
        red_add_u64(p.P + ((long long)t * kPCopies + (c % kPCopies)) * (E + 1) + e,
                    (1ull << kCountShift) + (unsigned long long)(v + kPOffset));
      }
    }
    if (range_err) atomicOr(p.err, MOE_DEVERR_RANGE);
  }

  // ---- the router sums, kFewPairs (token, entry) pairs at a time per thread
  bool bad = false, nan_seen = false;
  {
    const int npairs = T * (E + 1);
    for (int pb = tid; pb < npairs && !bad; pb += kFewPairs * kDecThreads) {
      unsigned long long w[kFewPairs][kPCopies];
      const unsigned long long* src[kFewPairs];
#pragma unroll
      for (int i = 0; i < kFewPairs; ++i) {
        const int pp = pb + i * kDecThreads;
        const int t = pp / (E + 1), e = pp - t * (E + 1);
        src[i] = p.P + (long long)t * kPCopies * (E + 1) + e;
#pragma unroll
        for (int q = 0; q < kPCopies; ++q)
          w[i][q] = (pp < npairs) ? ld_relaxed_u64(src[i] + q * (E + 1)) : 0ull;
      }
      uint64_t t0 = 0;
      uint32_t n = 0;
      for (;;) {
        unsigned pend = 0;
#pragma unroll
        for (int i = 0; i < kFewPairs; ++i) {
          if (pb + i * kDecThreads >= npairs) continue;
#pragma unroll
          for (int q = 0; q < kPCopies; ++q) {
            const unsigned want = (G > q) ? (unsigned)((G - q + kPCopies - 1) / kPCopies) : 0u;
            if ((unsigned)(w[i][q] >> kCountShift) != want) pend |= 1u << (i * kPCopies + q);
          }
        }
        if (!pend) break;
        if (poll_give_up(p, t0, n)) {
          bad = true;
          break;
        }
#pragma unroll
        for (int i = 0; i < kFewPairs; ++i)
#pragma unroll
          for (int q = 0; q < kPCopies; ++q)
            if ((pend >> (i * kPCopies + q)) & 1u) w[i][q] = ld_relaxed_u64(src[i] + q * (E + 1));
      }
      if (bad) break;
#pragma unroll
      for (int i = 0; i < kFewPairs; ++i) {
        const int pp = pb + i * kDecThreads;
        if (pp >= npairs) continue;
        const int t = pp / (E + 1), e = pp - t * (E + 1);
        long long sum = 0;
#pragma unroll
        for (int q = 0; q < kPCopies; ++q) {
          const long long cnt = (long long)(w[i][q] >> kCountShift);
          sum += (long long)(w[i][q] & ((1ull << kCountShift) - 1ull)) - cnt * kPOffset;
        }
        float v = unfix32(sum);
        if (e < E) {
          if (p.bias) v += __ldg(p.bias + e);
          if (c == 0) p.logits[(long long)t * E + e] = v;
          float kv = v;
          if (v != v) {
            nan_seen = true;
            kv = -INFINITY;
          }
          keys[t * 32 * ((E + 31) >> 5) + e] = ((unsigned long long)ord_key(kv) << 32) |
                                                 (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
        }
        lg[t * (E + 1) + e] = v;
      }
    }
  }
  if (tid < kMaxE / 32) umask[tid] = 0u;
  for (int i = tid; i < kFewUnion * kFewMax; i += kDecThreads) uslot[i] = (int8_t)-1;
  {
    const int nkey = 32 * ((E + 31) >> 5);
    for (int i = tid; i < T * nkey; i += kDecThreads)
      if (i % nkey >= E) keys[i] = 0ull;
    for (int i = tid; i < T * ((E + 31) >> 5) * k; i += kDecThreads) cand[i] = 0ull;
  }
  if (__syncthreads_or(bad)) {
    drain();
    return;
  }
  if (__syncthreads_or(nan_seen) && c == 0 && tid == 0) atomicOr(p.err, MOE_DEVERR_NAN_LOGIT);

  // ---- top-k of every token (up to 256 experts: warp t takes token t, lane l
  //      experts 8l .. 8l+7; else over the whole CTA); routing weights and
  //      shared gate of token t by warp t
  if (E <= 256) {
    if (warp < T) {
      const int nkey = 32 * ((E + 31) >> 5);
      const unsigned long long* kt = keys + warp * nkey;
      unsigned long long s8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = (8 * lane + i < nkey) ? kt[8 * lane + i] : 0ull;
      const unsigned long long kw = warp_topk_lists(s8, k, lane);
      if (lane < k) sel_e[warp * kMaxK + lane] = (int)(0xFFFFFFFFu - (uint32_t)kw);
    }
    __syncthreads();
  } else {
    cta_topk(keys, cand, E, k, T, sel_e, tid);
  }
  if (warp < T) {
    const float* lt = lg + warp * (E + 1);
    const int* se = sel_e + warp * kMaxK;
    // softmax over the k chosen logits in double-float arithmetic (within
    // one ulp of fp64), as in the decode kernel
    const int my_e = (lane < k) ? se[lane] : 0;
    float my_v = (lane < k) ? lt[my_e] : -INFINITY;
    if (my_v != my_v) my_v = -INFINITY;
    float top = lt[se[0]];
    if (top != top) top = -INFINITY;
    const dflt ex = (lane < k) ? df_softmax_term(my_v, top) : dflt{0.0f, 0.0f};
    dflt den = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const dflt ot = {__shfl_xor_sync(0xffffffffu, den.hi, o),
                       __shfl_xor_sync(0xffffffffu, den.lo, o)};
      den = df_add(den, ot);
    }
    if (lane < k) sel_w[warp * kMaxK + lane] = df_div(ex, den).hi;
    if (lane == 0) sig[warp] = p.has_shared ? 1.0f / (1.0f + expf(-lt[E])) : 0.0f;
  }
  __syncthreads();

  // ---- the union of the chosen experts, ascending (after the shared expert)
  for (int a = tid; a < T * k; a += kDecThreads) {
    const int e = sel_e[(a / k) * kMaxK + a % k];
    atomicOr(&umask[e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  if (warp == 0) {
    const int cnt = (lane < kMaxE / 32) ? __popc(umask[lane]) : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < kMaxE / 32) ubase[lane] = incl - cnt + p.has_shared;
    if (lane == 31) misc[0] = incl + p.has_shared;
  }
  __syncthreads();
  for (int a = tid; a < T * k; a += kDecThreads) {
    const int t = a / k, j = a - t * k;
    const int e = sel_e[t * kMaxK + j];
    const int u = ubase[e >> 5] + __popc(umask[e >> 5] & ((1u << (e & 31)) - 1u));
    ulist[u] = e;
    uslot[u * kFewMax + t] = (int8_t)j;
  }
  if (p.has_shared) {
    if (tid < T) uslot[tid] = (int8_t)k;
    if (tid == 0) ulist[0] = E;
  }
  __syncthreads();
  const int NB = misc[0] * bpe;
  const uint32_t ptag = (p.epoch << 6) | 0x80000000u;

  // ---- the CTA's blocks
  if (!pre && c < NB) {
    if (lane == 0) issue_gu(c, ulist[c / bpe]);
    if (tid == kDnTid) issue_dn(c, ulist[c / bpe]);
  }
  for (int b = c; b < NB; b += G) {
    const int u = b / bpe, blk = b - u * bpe;
    unsigned tmask = 0u;
    for (int t = 0; t < T; ++t)
      if (uslot[u * kFewMax + t] >= 0) tmask |= 1u << t;
    if (!copy_wait(p, bar0 + 8 * warp, ph_gu)) {
      drain();
      return;
    }
    if (lane == 0) infl[warp] = -1;
    ph_gu ^= 1;
    {
      const uint8_t* ub0 = gu_buf + (size_t)warp * kUnitsPerWarp * gu_unit;
      // one token at a time (compact code: each phase of this kernel runs
      // once per launch, so its instructions are fetched cold)
      for (unsigned m = tmask; m; m &= m - 1u) {
        const int t = __ffs(m) - 1;
        float acc[1][4];
        gateup_rows<1>(ub0, gu_unit, d, ng, xq + (size_t)t * 8 * ng, xsc + t * ng, xg + t * ng, 0,
                       0, 1u, lane, acc);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float gv = warp_sum(acc[0][2 * q]), uv = warp_sum(acc[0][2 * q + 1]);
          if (lane == 0) hb[t * kBlk + warp * kUnitsPerWarp + q] = gv / (1.0f + expf(-gv)) * uv;
        }
      }
    }
    // this warp's rows are used: the next block's rows for it load now
    if (b + G < NB && lane == 0) issue_gu(b + G, ulist[(b + G) / bpe]);
    __syncthreads();
    if (warp < T && ((tmask >> warp) & 1u))
      quant_h32(hb[warp * kBlk + lane], qt + warp * kBlk, hpk + warp * (kBlk / 8), &hsc[warp],
                &hsum[warp], lane);
    if (!copy_wait(p, dn_bar, ph_dn)) {
      drain();
      return;
    }
    if (tid == kDnTid) infl[kDnBar] = -1;
    ph_dn ^= 1;
    __syncthreads();
    {
      const unsigned long long tg = (unsigned long long)ptag << 32;
      for (int f = tid; f < d; f += kDecThreads) {
        const uint4 cw = dnc[f];
        const uint32_t sb = dnsb[f];
        for (unsigned m = tmask; m; m &= m - 1u) {
          const int t = __ffs(m) - 1;
          const int j = uslot[u * kFewMax + t];
          const float wj = (j < k) ? sel_w[t * kMaxK + j] : sig[t];
          const uint4* ht = hpk + t * (kBlk / 8);
          const float v = down_value(cw, sb, ht[0], ht[1], ht[2], ht[3], hsc[t], hsum[t], wj);
          st_relaxed_u64(p.part + (((long long)t * k1 + j) * bpe + blk) * d + f,
                         tg | __float_as_uint(v));
        }
      }
    }
    __syncthreads();  // the down columns and h are no longer read
    if (b + G < NB && tid == kDnTid) issue_dn(b + G, ulist[(b + G) / bpe]);
  }

  // ---- owned outputs of every token: the fixed-order sum of its partials
  //      (the decode kernel's order), two tokens' loads in flight together
  const int npart = k1 * bpe;
  for (int t0 = 0; t0 < T; t0 += 2) {
    const int nt = min(2, T - t0);
    for (int fl0 = 0; fl0 < nf; fl0 += 16) {
      const int fl = fl0 + (tid & 15), ch = tid >> 4;
      float s2[2] = {0.f, 0.f};
      if (fl < nf) {
        const unsigned long long* pf[2];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
          pf[tt] = p.part + (long long)(t0 + (tt < nt ? tt : 0)) * npart * d + f0 + fl;
        for (int bp = ch; bp < npart && !bad; bp += kRedChunks * kPollMax) {
          unsigned long long v[2][kPollMax];
#pragma unroll
          for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int i = 0; i < kPollMax; ++i) {
              const int bb = bp + i * kRedChunks;
              v[tt][i] = (bb < npart && tt < nt) ? ld_relaxed_u64(pf[tt] + (long long)bb * d)
                                                 : ((unsigned long long)ptag << 32);
            }
          uint64_t tw = 0;
          uint32_t n = 0;
          for (;;) {
            unsigned pend = 0;
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
              for (int i = 0; i < kPollMax; ++i)
                if ((uint32_t)(v[tt][i] >> 32) != ptag) pend |= 1u << (tt * kPollMax + i);
            if (!pend) break;
            if (poll_give_up(p, tw, n)) {
              bad = true;
              break;
            }
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
              for (int i = 0; i < kPollMax; ++i)
                if ((pend >> (tt * kPollMax + i)) & 1u)
                  v[tt][i] = ld_relaxed_u64(pf[tt] + (long long)(bp + i * kRedChunks) * d);
          }
#pragma unroll
          for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int i = 0; i < kPollMax; ++i)
              if (bp + i * kRedChunks < npart) s2[tt] += __uint_as_float((uint32_t)v[tt][i]);
        }
      }
      red2[ch * 16 + (tid & 15)] = s2[0];
      red2[(kRedChunks + ch) * 16 + (tid & 15)] = s2[1];
      if (__syncthreads_or(bad)) {
        drain();
        return;
      }
      if (tid < 32) {
        const int tt = tid >> 4, fo = tid & 15;
        if (tt < nt && fl0 + fo < nf) {
          float o = 0.f;
          for (int q = 0; q < kRedChunks; ++q) o += red2[(tt * kRedChunks + q) * 16 + fo];
          p.y[(long long)(t0 + tt) * d + f0 + fl0 + fo] =
              __bfloat16_as_ushort(__float2bfloat16_rn(o));
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

size_t decode_scratch_bytes(const Handle* h, int L) {
  const moe_config& c = h->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const size_t NB = (size_t)k1 * c.I / kBlk;
  auto r256 = [](size_t b) { return (b + 255) / 256 * 256; };
  return 256 + r256((size_t)2 * c.d * 4) + r256((size_t)L * kPCopies * (c.E + 1) * 8) +
         r256(NB * c.d * 8) + r256((size_t)L * c.E * 4) + r256((size_t)L * 4) + 256;
}

cudaError_t launch_decode(Handle* const* layers, int L, const uint16_t* x, const float* bias,
                          float eps, uint16_t* y, const moe_decode_trace* trace,
                          cudaStream_t st) {
  Handle* h0 = layers[0];
  const moe_config& c = h0->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const int G = h0->num_sms;
  if ((G + kPCopies - 1) / kPCopies > kMaxPerCopy) return cudaErrorInvalidConfiguration;
  const int nf_max = (c.d + G - 1) / G;
  const int NB = k1 * c.I / kBlk;
  const int Ep = decode_router_pitch(c.E);
  const DecSmem sm = dec_smem(c.d, c.E, Ep, nf_max);
  if (sm.total > 227 * 1024) return cudaErrorInvalidConfiguration;
  static_assert(sizeof(DecParams) < 32000, "kernel parameter size");
  uint8_t* scr = reinterpret_cast<uint8_t*>(h0->ws.logit_part);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  auto r256 = [](size_t b) { return (b + 255) / 256 * 256; };
  // scratch: [abort | out | P] (zeroed before every launch) | partials | logits | sigma
  for (int l0 = 0; l0 < L; l0 += kMaxDecLayers) {
    const int nl = (L - l0) < kMaxDecLayers ? (L - l0) : kMaxDecLayers;
    uint8_t* q = scr;
    int* abort_flag = reinterpret_cast<int*>(q);
    q += 256;
    uint32_t* out = reinterpret_cast<uint32_t*>(q);
    q += r256((size_t)2 * c.d * 4);
    unsigned long long* P = reinterpret_cast<unsigned long long*>(q);
    const size_t zero_bytes = (size_t)(q - scr) + (size_t)nl * kPCopies * (c.E + 1) * 8;
    q += r256((size_t)kMaxDecLayers * kPCopies * (c.E + 1) * 8);
    unsigned long long* part = reinterpret_cast<unsigned long long*>(q);
    q += r256((size_t)NB * c.d * 8);
    float* logits_s = reinterpret_cast<float*>(q);
    q += r256((size_t)kMaxDecLayers * c.E * 4);
    float* sigma_s = reinterpret_cast<float*>(q);
    DecParams p;
    for (int i = 0; i < nl; ++i) {
      const Handle* h = layers[l0 + i];
      p.layer[i].gu = h->dc_gu;
      p.layer[i].dnc = h->dc_dn;
      p.layer[i].dnsb =
          reinterpret_cast<const uint32_t*>(h->dc_dn + (size_t)h->n_exp * c.I / 2 * c.d);
      p.layer[i].w_rt = h->dc_router_t;
    }
    p.L = nl;
    p.d = c.d;
    p.E = c.E;
    p.k = c.k;
    p.I = c.I;
    p.has_shared = c.has_shared;
    p.Ep = Ep;
    p.nf_max = nf_max;
    p.NB = NB;
    p.epoch = ++h0->dec_epoch;
    p.x = (l0 == 0) ? x : y;
    p.norm_first = (l0 == 0) ? 0 : 1;
    p.bias = bias ? bias + (long long)l0 * c.E : nullptr;
    p.eps = eps;
    p.y = y;
    p.abort_flag = abort_flag;
    p.P = P;
    p.part = part;
    p.out = out;
    p.logits = (trace && trace->logits) ? trace->logits + (long long)l0 * c.E : logits_s;
    p.sigma = (trace && trace->sigma) ? trace->sigma + l0 : sigma_s;
    p.tr_idx = (trace && trace->idx) ? trace->idx + (long long)l0 * c.k : nullptr;
    p.tr_w = (trace && trace->w) ? trace->w + (long long)l0 * c.k : nullptr;
    p.tr_out = (trace && trace->out)
                   ? reinterpret_cast<uint16_t*>(trace->out) + (long long)l0 * c.d
                   : nullptr;
    p.tr_ns = (trace && trace->timestamps) ? trace->timestamps + (long long)l0 * 4 : nullptr;
    p.err = h0->dev_err;
    p.wait_ns = h0->wait_ns;
    p.unset_flag = h0->test_unset_flag;
    // the abort flag, the tagged outputs and the router sums start at zero
    cudaError_t e = cudaMemsetAsync(scr, 0, zero_bytes, st);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    e = cudaLaunchCooperativeKernel((const void*)decode_kernel, dim3(G), dim3(kDecThreads), args,
                                    sm.total, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t few_scratch_bytes(const Handle* h) {
  const moe_config& c = h->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  auto r256 = [](size_t b) { return (b + 255) / 256 * 256; };
  return 256 + r256((size_t)kFewMax * kPCopies * (c.E + 1) * 8) +
         r256((size_t)kFewMax * k1 * (c.I / kBlk) * c.d * 8);
}

int few_max_tokens() { return kFewMax; }

bool few_supported(const Handle* h, int T) {
  const moe_config& c = h->cfg;
  // the logits go to the workspace's [max_tokens][E] rows
  if (T < 2 || T > kFewMax || T > c.max_tokens || !h->ws.few) return false;
  const int G = h->num_sms;
  if ((G + kPCopies - 1) / kPCopies > kMaxPerCopy) return false;
  const int nf_max = (c.d + G - 1) / G;
  return few_smem(T, c.d, c.E, decode_router_pitch(c.E), nf_max).total <= 227 * 1024;
}

cudaError_t launch_few(Handle* h, const uint16_t* x, int T, const float* bias, uint16_t* y,
                       cudaStream_t st) {
  const moe_config& c = h->cfg;
  const int G = h->num_sms;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const int nf_max = (c.d + G - 1) / G;
  const int Ep = decode_router_pitch(c.E);
  const FewSmem sm = few_smem(T, c.d, c.E, Ep, nf_max);
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(few_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  auto r256 = [](size_t b) { return (b + 255) / 256 * 256; };
  // scratch: [abort | P] (zeroed before every launch) | partials
  uint8_t* q = h->ws.few;
  int* abort_flag = reinterpret_cast<int*>(q);
  unsigned long long* P = reinterpret_cast<unsigned long long*>(q + 256);
  const size_t zero_bytes = 256 + (size_t)T * kPCopies * (c.E + 1) * 8;
  unsigned long long* part = reinterpret_cast<unsigned long long*>(
      q + 256 + r256((size_t)kFewMax * kPCopies * (c.E + 1) * 8));
  (void)k1;
  FewParams p;
  p.W.gu = h->dc_gu;
  p.W.dnc = h->dc_dn;
  p.W.dnsb = reinterpret_cast<const uint32_t*>(h->dc_dn + (size_t)h->n_exp * c.I / 2 * c.d);
  p.W.w_rt = h->dc_router_t;
  p.T = T;
  p.d = c.d;
  p.E = c.E;
  p.k = c.k;
  p.I = c.I;
  p.has_shared = c.has_shared;
  p.Ep = Ep;
  p.nf_max = nf_max;
  p.epoch = ++h->dec_epoch;
  p.x = x;
  p.bias = bias;
  p.y = y;
  p.logits = h->ws.logits;
  p.part = part;
  p.P = P;
  p.abort_flag = abort_flag;
  p.err = h->dev_err;
  p.wait_ns = h->wait_ns;
  cudaError_t e = cudaMemsetAsync(q, 0, zero_bytes, st);
  if (e != cudaSuccess) return e;
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel((const void*)few_kernel, dim3(G), dim3(kDecThreads), args,
                                     sm.total, st);
}

}  // namespace moe
