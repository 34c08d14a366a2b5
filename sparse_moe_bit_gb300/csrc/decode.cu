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
// Two grid-wide barriers per layer:
//   A : every CTA reads the previous output out_{l-1} and the router sums P_l
//       in one pass, folds 1/rms(out_{l-1}) into the logits (the rest of the
//       layer works on the unnormalised vector and scales its dot products),
//       repeats the top-k selection in one warp and issues the bulk copies of
//       its block's gate/up rows and down columns straight after it.
//   B : gate/up of the block (two features per warp), h of the block to
//       16-bit integers, the block's partial over all d outputs -> global
//       -> grid barrier
//   R : out[f] = sum over blocks of the partials (fixed order) for the owned
//       features, rounded to bf16; then the next layer's router partial sums
//       over those features: P_{l+1}[e] += sum_f out[f] W_r'[e][f],
//       accumulated as 64-bit fixed-point integers (2^-32 units) into one of
//       several copies of P (so that fewer CTAs meet on one address); integer
//       addition makes the sum exact and independent of the order of
//       arrival -> grid barrier
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

namespace moe {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kBlk = 32;                        // intermediate features per block
constexpr int kUnitsPerWarp = kBlk / kDecWarps;  // gate/up features a warp computes
static_assert(kUnitsPerWarp == 2, "gate/up takes two features per warp");
constexpr int kMaxDecLayers = 64;
constexpr int kPCopies = 8;  // copies of the router sums: CTA c adds into copy c % kPCopies
constexpr int kPSlots = 3;   // layer l's sums live in slot l % kPSlots
constexpr int kRedChunks = 32;  // partial sums per owned feature in the reduction
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;
constexpr float kFix = 4294967296.0f;  // 2^32

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
  float* part;          // [NB][d] the blocks' weighted partial outputs
  uint16_t* out;        // [2][d]: layer l writes row l % 2
  unsigned long long* P;  // [kPSlots][kPCopies][E+1] fixed-point router sums, zero at launch
  unsigned* bar;        // grid barrier arrivals, zero at launch
  int* abort_flag;      // zero at launch
  int* err;
};

// shared-memory carve-up (the host sizes the launch with the same function)
struct DecSmem {
  size_t xq, xsc, xg, gu, dnc, dnsb, hb, hpk, rt, outs, red2, lg, lb, sel_e, sel_w, misc, red,
      infl, bars, ok, total;
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
  s.xq = dec_take(o, (size_t)d * 2, 16);
  s.xsc = dec_take(o, (size_t)(d / 64) * 4, 16);
  s.xg = dec_take(o, (size_t)(d / 64) * 4, 16);
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
  s.sel_e = dec_take(o, kMaxK * 4, 16);
  s.sel_w = dec_take(o, kMaxK * 4, 16);
  s.misc = dec_take(o, 16, 16);
  s.red = dec_take(o, kDecWarps * 4, 16);
  s.infl = dec_take(o, (kDecWarps + 2) * 4, 16);
  s.bars = dec_take(o, (kDecWarps + 3) * 8, 8);
  s.ok = dec_take(o, 16, 16);
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

// order-preserving key of a float (larger value, larger key); -0 taken as +0
__device__ __forceinline__ uint32_t ord_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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
// group maximum.  (e >= -127 keeps 2^-e a normal float; smaller groups are
// below 2^-114 everywhere.)
__device__ __forceinline__ int group_exponent(float amax) {
  const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;  // floor(log2 amax)
  return max(ex - 13, -127);
}
// 2^-e for a group exponent e
__device__ __forceinline__ float inv_pow2(int e) { return __int_as_float((127 - e) << 23); }
// 2^e, exact also where it is subnormal (two power-of-two factors)
__device__ __forceinline__ float pow2(int e) {
  const int a = e >> 1, b = e - a;
  return __int_as_float((a + 127) << 23) * __int_as_float((b + 127) << 23);
}
// fp32 bits whose low 16 bits are round(v * 2^-e) as a 16-bit integer:
// adding 1.5 * 2^23 leaves the rounded integer in the low mantissa bits
__device__ __forceinline__ uint32_t quant_bits(float v, float inv) {
  return __float_as_uint(fmaf(v, inv, 12582912.0f));
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


// Top-k of lg[0..E) in one warp, ranked by (value descending, index
// ascending), NaN taken as -inf.  Lane l holds the experts l, l+32, ... as
// 64-bit keys (order key << 32 | ~index), sorts them (bitonic network) and
// then each round needs only the head of every lane: the warp maximum of the
// high words, then of the low words among the lanes that hold it, names the
// winner, whose lane drops its head.  sel_e[r] = the r-th choice (lane 0
// writes it).
template <int VPL>
__device__ __forceinline__ void warp_topk(const float* lg, int E, int k, int lane, int* sel_e,
                                          bool* nan_seen) {
  unsigned long long K[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    unsigned long long key = 0ull;  // empty; every real key is larger
    if (e < E) {
      float v = lg[e];
      if (v != v) {
        v = -INFINITY;
        *nan_seen = true;
      }
      key = ((unsigned long long)ord_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
    }
    K[j] = key;
  }
#pragma unroll
  for (int size = 2; size <= VPL; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = K[i], b = K[j];
          const bool sw = desc ? (a < b) : (a > b);
          K[i] = sw ? b : a;
          K[j] = sw ? a : b;
        }
      }
    }
  }
  for (int r = 0; r < k; ++r) {
    const uint32_t hi = (uint32_t)(K[0] >> 32), lo = (uint32_t)K[0];
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    if (hi == mh && lo == ml) {
#pragma unroll
      for (int j = 0; j + 1 < VPL; ++j) K[j] = K[j + 1];
      K[VPL - 1] = 0ull;
    }
    if (lane == 0) sel_e[r] = (int)(0xFFFFFFFFu - ml);
  }
}

// Grid-wide barrier number n (0-based): arrivals are counted monotonically, so
// barrier n completes at (n + 1) * gridDim.x.  The arrival is a release and
// the poll an acquire at GPU scope, which orders every CTA's writes before the
// barrier (its threads meet at __syncthreads first) with every read after it.
// Bounded: on time-out (or when another CTA gave up) every CTA leaves.
__device__ bool grid_sync(const DecParams& p, unsigned n, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p.bar), "r"(1u) : "memory");
    const unsigned target = (n + 1) * gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.bar) : "memory");
      if (v >= target) break;
      if ((i & 15u) == 15u) {
        if (*(volatile int*)p.abort_flag) {
          ok = 0;
          break;
        }
        if (globaltimer_ns() - t0 > kWaitNs) {
          atomicOr(p.err, MOE_DEVERR_GRID_TIMEOUT);
          atomicExch(p.abort_flag, 1);
          ok = 0;
          break;
        }
      }
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Bounded wait on an mbarrier phase; the thread sleeps in hardware between
// checks.  On time-out (or when another CTA gave up) records the error.
__device__ __forceinline__ bool copy_wait(const DecParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*(volatile int*)p.abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(p.err, MOE_DEVERR_WAIT_TIMEOUT);
      atomicExch(p.abort_flag, 1);
      return false;
    }
  }
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
  const DecSmem L = dec_smem(d, E, Ep, p.nf_max);
  uint4* xq = reinterpret_cast<uint4*>(dsm + L.xq);   // [8 words][ng] packed int16 x
  float* xsc = reinterpret_cast<float*>(dsm + L.xsc);  // [ng] scale of a group of x
  float* xg = reinterpret_cast<float*>(dsm + L.xg);    // [ng] sum of a group of x
  uint8_t* gu_buf = dsm + L.gu;                        // [32 units] of d + d/8 bytes
  const uint4* dnc = reinterpret_cast<const uint4*>(dsm + L.dnc);        // [d] block codes
  const uint32_t* dnsb = reinterpret_cast<const uint32_t*>(dsm + L.dnsb);  // [d] s,b words
  float* hb = reinterpret_cast<float*>(dsm + L.hb);    // [32] h of the block
  uint4* hpk = reinterpret_cast<uint4*>(dsm + L.hpk);  // [4 words] packed int16 h
  const uint16_t* rt_buf = reinterpret_cast<const uint16_t*>(dsm + L.rt);
  float* outs = reinterpret_cast<float*>(dsm + L.outs);
  float* red2 = reinterpret_cast<float*>(dsm + L.red2);  // [chunks][16] reduction partials
  float* lg = reinterpret_cast<float*>(dsm + L.lg);  // raw sums, then logits; [E]: shared gate
  float* lb = reinterpret_cast<float*>(dsm + L.lb);  // logit bias
  int* sel_e = reinterpret_cast<int*>(dsm + L.sel_e);
  float* sel_w = reinterpret_cast<float*>(dsm + L.sel_w);
  float* misc = reinterpret_cast<float*>(dsm + L.misc);  // [0] sigma [1] 1/rms [2] h scale [3] h sum
  float* red = reinterpret_cast<float*>(dsm + L.red);
  // parity of the copies in flight on each mbarrier (-1: none), for the
  // bounded drain on the error path
  volatile int* infl = reinterpret_cast<volatile int*>(dsm + L.infl);
  const uint32_t bar0 = smem_u32(dsm + L.bars);  // [warps] gate/up, then down, router
  int* s_ok = reinterpret_cast<int*>(dsm + L.ok);
  const int kDnBar = kDecWarps, kRtBar = kDecWarps + 1;
  const uint32_t dn_bar = bar0 + 8 * kDnBar;
  const uint32_t rt_bar = bar0 + 8 * kRtBar;
  const uint32_t route_bar = bar0 + 8 * (kDecWarps + 2);  // the top-k of the layer is known
  const int wwarp = kDecWarps - 1;  // computes the routing weights

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int f0 = (int)((long long)c * d / G), f1 = (int)((long long)(c + 1) * d / G);
  const int nf = f1 - f0;
  const int gu_unit = d + d / 8;

  if (tid == 0) {
    for (int i = 0; i < kDecWarps + 3; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (tid < kDecWarps + 2) infl[tid] = -1;
  __syncthreads();
  uint32_t ph_gu = 0, ph_dn = 0, ph_rt = 0, ph_route = 0;
  unsigned nsync = 0;

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
  // (b % bpe) * 32 .. + 31.  Issue its bulk copies: lane i < 16 the gate/up
  // rows of warp i's two features, lane 16 the block's down columns (codes
  // of every output row, then the rows' scale/bias words of its input
  // group).  Called by every lane of one warp.
  auto issue_block = [&](int b, const DecLayer& W) {
    const int j = b / bpe, i0 = (b - j * bpe) * kBlk;
    const long long ex = (j < k) ? sel_e[j] : E;
    if (lane < kDecWarps) {
      const uint32_t bar = bar0 + 8 * lane;
      const uint32_t bytes = (uint32_t)(kUnitsPerWarp * gu_unit);
      infl[lane] = (int)ph_gu;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(gu_buf + (size_t)lane * kUnitsPerWarp * gu_unit),
               W.gu + (ex * I + i0 + lane * kUnitsPerWarp) * gu_unit, bytes, bar);
    } else if (lane == kDecWarps) {
      infl[kDnBar] = (int)ph_dn;
      mbar_arrive_expect_tx(dn_bar, (uint32_t)(d * 20));
      bulk_g2s(smem_u32(dsm + L.dnc), W.dnc + (ex * bpe + i0 / kBlk) * (long long)d * 16,
               (uint32_t)(d * 16), dn_bar);
      bulk_g2s(smem_u32(dsm + L.dnsb), W.dnsb + (ex * (I / 64) + i0 / 64) * (long long)d,
               (uint32_t)(d * 4), dn_bar);
    }
  };

  // Four consecutive activations v0..v3 at index i0 (a multiple of 4; the 16
  // lanes of a half-warp hold one group of 64) -> 16-bit integers with the
  // group's power-of-two scale, stored as the packed pairs the integer dot
  // products take: word m of group g holds (x0,x2), (x4,x6), (x1,x3),
  // (x5,x7) of K indices 8m..8m+7.  Also the group's scale and sum.  Every
  // lane of the warp takes part (shuffles); act = false contributes nothing.
  auto quant_x4 = [&](float v0, float v1, float v2, float v3, int i0, bool act) {
    float am = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
    float sum = (v0 + v1) + (v2 + v3);
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    const int e = group_exponent(am);
    const float inv = inv_pow2(e);
    const uint32_t b0 = quant_bits(v0, inv), b1 = quant_bits(v1, inv);
    const uint32_t b2 = quant_bits(v2, inv), b3 = quant_bits(v3, inv);
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
  };

  // x (bf16 [d]) -> quantised activations in shared memory, with optional
  // RMS normalisation; also the owned features' values (used for the input
  // of the first layer of a launch).
  auto load_x = [&](const uint16_t* src, bool norm) {
    float r = 1.0f;
    if (norm) {
      float ss = 0.f;
      for (int i = tid; i < d; i += kDecThreads) {
        const float v = bf16f(__ldcg(src + i));
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
      if (act) raw = __ldcg(reinterpret_cast<const uint2*>(src + i0));
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

  // P_slot[copy c % kPCopies][e] += sum_{f owned} outs[f] * W'[e][f]
  // (e = E: the shared gate)
  auto router_partial = [&](int slot) {
    unsigned long long* Pq =
        p.P + ((long long)slot * kPCopies + (c % kPCopies)) * (long long)(E + 1);
    for (int e = tid; e <= E; e += kDecThreads) {
      float acc = 0.f;
      for (int f = 0; f < nf; ++f) acc = fmaf(outs[f], bf16f(rt_buf[f * Ep + e]), acc);
      atomicAdd(Pq + e, (unsigned long long)__float2ll_rn(acc * kFix));
    }
  };

  auto issue_router_copy = [&](int l) {
    if (tid == 32 && nf > 0) {  // lane 0 of warp 1
      const uint32_t bytes = (uint32_t)nf * Ep * 2;
      infl[kRtBar] = (int)ph_rt;
      mbar_arrive_expect_tx(rt_bar, bytes);
      bulk_g2s(smem_u32(dsm + L.rt), p.layer[l].w_rt + (long long)f0 * Ep, bytes, rt_bar);
    }
  };

  // ---- prologue: x_0 and the router sums of layer 0 (slot 0)
  issue_router_copy(0);
  load_x(p.x, p.norm_first != 0);
  if (nf > 0) {
    if (!copy_wait(p, rt_bar, ph_rt)) {
      drain();
      return;
    }
    if (tid == 0) infl[kRtBar] = -1;
  }
  ph_rt ^= 1;
  if (nf > 0) router_partial(0);
  if (!grid_sync(p, nsync++, s_ok)) {
    drain();
    return;
  }

  for (int l = 0; l < p.L; ++l) {
    const DecLayer& W = p.layer[l];
    stamp(p, l, 0);
    // ---- A: out_{l-1} and P_l in one pass; routing in warp 0; copies
    if (l + 1 < p.L) issue_router_copy(l + 1);
    // every load of this step is issued before any of them is used: the
    // router sums (expert e = tid), its bias, then the previous output
    const unsigned long long* Ps = p.P + (long long)(l % kPSlots) * kPCopies * (E + 1);
    unsigned long long pv[kPCopies];
    float be = 0.0f;
    if (tid <= E) {
#pragma unroll
      for (int q = 0; q < kPCopies; ++q) pv[q] = __ldcg(Ps + q * (E + 1) + tid);
      if (tid < E && p.bias) be = __ldg(p.bias + (long long)l * E + tid);
    }
    if (l > 0) {
      const uint16_t* src = p.out + (long long)((l - 1) & 1) * d;
      float ss = 0.f;
      for (int ib = 0; ib < d; ib += 4 * kDecThreads) {
        const int i0 = ib + 4 * tid;
        const bool act = i0 < d;
        uint2 raw = make_uint2(0u, 0u);
        if (act) raw = __ldcg(reinterpret_cast<const uint2*>(src + i0));
        const float v0 = bf16f(raw.x & 0xFFFFu), v1 = bf16f(raw.x >> 16);
        const float v2 = bf16f(raw.y & 0xFFFFu), v3 = bf16f(raw.y >> 16);
        ss = fmaf(v0, v0, ss);
        ss = fmaf(v1, v1, ss);
        ss = fmaf(v2, v2, ss);
        ss = fmaf(v3, v3, ss);
        quant_x4(v0, v1, v2, v3, i0, act);
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
    }
    {
      if (tid <= E) {
        long long sum = 0;
#pragma unroll
        for (int q = 0; q < kPCopies; ++q) sum += (long long)pv[q];
        lg[tid] = __ll2float_rn(sum) * (1.0f / 4294967296.0f);
        if (tid < E) lb[tid] = be;
      }
      for (int e = tid + kDecThreads; e <= E; e += kDecThreads) {  // E = 512 only
        long long sum = 0;
#pragma unroll
        for (int q = 0; q < kPCopies; ++q) sum += (long long)__ldcg(Ps + q * (E + 1) + e);
        lg[e] = __ll2float_rn(sum) * (1.0f / 4294967296.0f);
        if (e < E) lb[e] = p.bias ? p.bias[(long long)l * E + e] : 0.0f;
      }
      if (c == 0) {  // the slot of layer l-1 is free (read before the last barrier)
        unsigned long long* Pz =
            p.P + (long long)((l + kPSlots - 1) % kPSlots) * kPCopies * (E + 1);
        for (int i = tid; i < kPCopies * (E + 1); i += kDecThreads) Pz[i] = 0ull;
      }
    }
    __syncthreads();
    float r = 1.0f;  // 1/rms of out_{l-1} (x_0 is normalised already)
    if (l > 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) t += red[w];
      r = rsqrtf(t / (float)d + p.eps);
    }
    if (warp == 0) {
      for (int e = lane; e <= E; e += 32) {
        float v = lg[e] * r;
        if (e < E) {
          v += lb[e];
          lg[e] = v;
          if (c == 0) p.logits[(long long)l * E + e] = v;
        } else {
          const float sg = p.has_shared ? 1.0f / (1.0f + expf(-v)) : 0.0f;
          misc[0] = sg;
          if (c == 0) p.sigma[l] = sg;
        }
      }
      __syncwarp();
      bool nan_seen = false;
      if (E <= 256) warp_topk<8>(lg, E, k, lane, sel_e, &nan_seen);
      else warp_topk<kMaxE / 32>(lg, E, k, lane, sel_e, &nan_seen);
      if (__any_sync(0xffffffffu, nan_seen) && lane == 0 && c == 0)
        atomicOr(p.err, MOE_DEVERR_NAN_LOGIT);
      __syncwarp();
      if (c < NB) issue_block(c, W);
      if (lane == kDecWarps + 1) mbar_arrive(route_bar);  // sel_e and the logits are ready
      stamp(p, l, 1);
    }
    if (warp == wwarp) {
      // routing weights (softmax over the k chosen logits in double-float
      // arithmetic, within one ulp of fp64), off the path of the copies and
      // of the other warps' gate/up work
      if (!copy_wait(p, route_bar, ph_route)) {
        drain();
        return;
      }
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
    }
    ph_route ^= 1;

    // ---- B: the CTA's blocks: gate/up, h, and the block's partial output
    for (int b = c, nb = 0; b < NB; b += G, ++nb) {
      const int j = b / bpe;
      if (nb > 0) {
        __syncthreads();  // the previous block's buffers are no longer read
        if (warp == 0) issue_block(b, W);
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
        float ag[2] = {0.f, 0.f}, au[2] = {0.f, 0.f};
        for (int g = lane; g < ng; g += 32) {
          uint4 xw[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) xw[m] = xq[m * ng + g];
          const float sc = xsc[g], X = xg[g];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint8_t* ub = ub0 + t * gu_unit;
            const uint4 cg0 = *reinterpret_cast<const uint4*>(ub + g * 32);
            const uint4 cg1 = *reinterpret_cast<const uint4*>(ub + g * 32 + 16);
            const uint4 cu0 = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32);
            const uint4 cu1 = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32 + 16);
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
            const uint32_t sbg = reinterpret_cast<const uint32_t*>(ub + d)[g];
            const uint32_t sbu = reinterpret_cast<const uint32_t*>(ub + d + d / 16)[g];
            ag[t] += s_of(sbg) * (sc * (float)(pg0 + pg1)) + b_of(sbg) * X;
            au[t] += s_of(sbu) * (sc * (float)(pu0 + pu1)) + b_of(sbu) * X;
          }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float gv = warp_sum(ag[t]) * r, uv = warp_sum(au[t]) * r;
          if (lane == 0) hb[warp * kUnitsPerWarp + t] = gv / (1.0f + expf(-gv)) * uv;
        }
      }
      __syncthreads();
      // h of the block -> 16-bit integers with one power-of-two scale, packed
      // as the integer dot products take them (word m: features 8m..8m+7)
      if (warp == 0) {
        const float v = hb[lane];
        float am = fabsf(v), hs = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
          hs += __shfl_xor_sync(0xffffffffu, hs, o);
        }
        const int e = group_exponent(am);
        uint32_t* qt = reinterpret_cast<uint32_t*>(red2);
        qt[lane] = quant_bits(v, inv_pow2(e));
        __syncwarp();
        if (lane < kBlk / 8) {
          const uint32_t* q8 = qt + lane * 8;
          hpk[lane] = make_uint4(pack_lo16(q8[0], q8[2]), pack_lo16(q8[4], q8[6]),
                                 pack_lo16(q8[1], q8[3]), pack_lo16(q8[5], q8[7]));
        }
        if (lane == 0) {
          misc[2] = pow2(e);
          misc[3] = hs;
        }
      }
      if (!copy_wait(p, dn_bar, ph_dn)) {
        drain();
        return;
      }
      if (tid == 0) infl[kDnBar] = -1;
      ph_dn ^= 1;
      __syncthreads();
      // the block's partial output: part[b][f] = w_j (s sum_i q_i h_i + beta H)
      {
        const uint4 h0 = hpk[0], h1 = hpk[1], h2 = hpk[2], h3 = hpk[3];
        const float hsc = misc[2], Hs = misc[3];
        const float wj = (j < k) ? sel_w[j] : misc[0];
        float* pb = p.part + (long long)b * d;
        for (int f = tid; f < d; f += kDecThreads) {
          const uint4 cw = dnc[f];
          const uint32_t sb = dnsb[f];
          const int a = (dot8i(cw.x, h0, 0) + dot8i(cw.y, h1, 0)) +
                        (dot8i(cw.z, h2, 0) + dot8i(cw.w, h3, 0));
          pb[f] = wj * (s_of(sb) * (hsc * (float)a) + b_of(sb) * Hs);
        }
      }
    }

    // ---- every block's partial is in global memory
    if (!grid_sync(p, nsync++, s_ok)) {
      drain();
      return;
    }
    stamp(p, l, 2);
    // ---- R: out[f] = sum over blocks of part[b][f] (fixed order), bf16
    {
      uint16_t* outl = p.out + (long long)(l & 1) * d;
      for (int fl0 = 0; fl0 < nf; fl0 += 16) {
        const int fl = fl0 + (tid & 15), ch = tid >> 4;  // 32 chunks of blocks
        float s = 0.f;
        if (fl < nf) {
          const float* pf = p.part + f0 + fl;
#pragma unroll 4
          for (int b = ch; b < NB; b += kRedChunks) s += __ldcg(pf + (long long)b * d);
        }
        red2[ch * 16 + (tid & 15)] = s;
        __syncthreads();
        if (tid < 16 && fl0 + tid < nf) {
          float o = 0.f;
          for (int q = 0; q < kRedChunks; ++q) o += red2[q * 16 + tid];
          const uint16_t ob = __bfloat16_as_ushort(__float2bfloat16_rn(o));
          const int f = f0 + fl0 + tid;
          outs[fl0 + tid] = bf16f(ob);
          outl[f] = ob;
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
        if (tid == 0) infl[kRtBar] = -1;
      }
      ph_rt ^= 1;
      if (nf > 0) router_partial((l + 1) % kPSlots);
      if (!grid_sync(p, nsync++, s_ok)) {
        drain();
        return;
      }
    }
  }
}

}  // namespace

size_t decode_scratch_bytes(const Handle* h, int L) {
  const moe_config& c = h->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const size_t NB = (size_t)k1 * c.I / kBlk;
  return 256 + (size_t)kPSlots * kPCopies * (c.E + 1) * 8 + 256 + NB * c.d * 4 + 256 +
         (size_t)L * c.E * 4 + (size_t)L * 4 + 256 + (size_t)2 * c.d * 2 + 2048;
}

cudaError_t launch_decode(Handle* const* layers, int L, const uint16_t* x, const float* bias,
                          float eps, uint16_t* y, const moe_decode_trace* trace,
                          cudaStream_t st) {
  const Handle* h0 = layers[0];
  const moe_config& c = h0->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const int G = h0->num_sms;
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
  // scratch: [barrier, abort | P] (zeroed before every launch) | partials | logits | sigma | out
  uint8_t* q = scr;
  unsigned* bar = reinterpret_cast<unsigned*>(q);
  int* abort_flag = reinterpret_cast<int*>(q + 4);
  q += 256;
  unsigned long long* P = reinterpret_cast<unsigned long long*>(q);
  q += ((size_t)kPSlots * kPCopies * (c.E + 1) * 8 + 255) / 256 * 256;
  const size_t zero_bytes = (size_t)(q - scr);
  float* part = reinterpret_cast<float*>(q);
  q += ((size_t)NB * c.d * 4 + 255) / 256 * 256;
  float* logits_s = reinterpret_cast<float*>(q);
  q += (size_t)kMaxDecLayers * c.E * 4;
  float* sigma_s = reinterpret_cast<float*>(q);
  q += (size_t)kMaxDecLayers * 4 + 256;
  uint16_t* out = reinterpret_cast<uint16_t*>(q);
  for (int l0 = 0; l0 < L; l0 += kMaxDecLayers) {
    const int nl = (L - l0) < kMaxDecLayers ? (L - l0) : kMaxDecLayers;
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
    p.x = (l0 == 0) ? x : y;
    p.norm_first = (l0 == 0) ? 0 : 1;
    p.bias = bias ? bias + (long long)l0 * c.E : nullptr;
    p.eps = eps;
    p.y = y;
    p.bar = bar;
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
    // the barrier counter, the abort flag and the router sums start at zero
    cudaError_t e = cudaMemsetAsync(scr, 0, zero_bytes, st);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    e = cudaLaunchCooperativeKernel((const void*)decode_kernel, dim3(G), dim3(kDecThreads), args,
                                    sm.total, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
