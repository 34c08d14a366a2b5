// Batch-1 decode path: one persistent cooperative kernel runs every layer of
// the chain on CUDA cores.  The work is bound by weight reads (4.5 bits per
// weight): each CTA streams only its share of the selected experts' rows into
// shared memory with bulk (TMA) copies issued as soon as the routing is known,
// and computes while they land.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Optimizing the one-row weight path" (a row-parallel GEMV: a SIMD group
// cooperates on one output while reading different parts of the weight
// matrix), §"Reduce intermediate and state traffic" (gate and up projections
// fused with their gated activation; the output projection fused with its
// routing score and the shared expert's result) and §"Keep each decode step
// on the GPU" (no host synchronisation between steps).
//
// Two grid-wide barriers per layer.  CTA c owns output features
// [c*d/G, (c+1)*d/G) and a contiguous range of the (slot j, feature f) units
// of the k+1 active experts.
//   A : every CTA rebuilds x_l = out_{l-1} / sqrt(mean(out_{l-1}^2) + eps)
//       from the previous output, turns the router sums P_l into logits
//       (times the same 1/rms), repeats the top-k selection, and issues the
//       bulk copies of its gate/up rows and its down rows.
//   GU: h_j[f] = silu(G_j[f] . x) * (U_j[f] . x) for the owned units -> global
//       -> grid barrier
//   D : out[f] = sum_j w_j (D_j[f] . h_j) + sigma (D_s[f] . h_s) for the owned
//       features (fixed order), then the next layer's router partial sums over
//       those features: P_{l+1}[e] += sum_f out[f] W_r'[e][f], accumulated as
//       64-bit fixed-point integers (2^-32 units), so the sum is exact and does
//       not depend on the order of arrival -> grid barrier
// Dot products use the split s*q + beta per 64-group:
//   sum_i (s q_i + beta) x_i = s (sum_i (128 + q_i) x_i - 128 X) + beta X,
// X = sum_i x_i, with the code turned into the fp32 value 128 + q by one byte
// permute (exponent byte 0x43, code in the top mantissa byte).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxDecLayers = 64;
constexpr int kMaxUnitsPerWarp = 4;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kFix = 4294967296.0f;  // 2^32

struct DecLayer {
  const uint8_t* gu_codes;  // [n_exp][2I][d/2]
  const uint32_t* gu_sb;    // [n_exp][2I][d/64]
  const uint8_t* dn_codes;  // [n_exp][d][I/2]
  const uint32_t* dn_sb;    // [n_exp][d][sbp]
  const uint16_t* w_rt;     // [d][Ep] router transposed + shared-gate column
};

struct DecParams {
  DecLayer layer[kMaxDecLayers];
  int L, d, E, k, I, has_shared, Ep;
  int nf_max, upw;  // output features per CTA (max), units per warp (max)
  int sbp;          // 32-bit scale/bias words per down row (padded)
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
  float* H;             // [k1][I]
  uint16_t* out;        // [d]
  unsigned long long* P;  // [L][E+1] fixed-point router sums, zero at launch
  unsigned* bar;        // grid barrier arrivals, zero at launch
  int* abort_flag;      // zero at launch
  int* err;
};

// shared-memory carve-up (the host sizes the launch with the same function)
struct DecSmem {
  size_t xs2, xg, hs2, hw, gu, dn, rt, outs, lg, sel_e, sel_w, misc, red, bars, ok, total;
};
__host__ __device__ inline size_t dec_take(size_t& o, size_t bytes, size_t align) {
  o = (o + align - 1) / align * align;
  const size_t r = o;
  o += bytes;
  return r;
}
__host__ __device__ inline DecSmem dec_smem(int d, int I, int k1, int E, int Ep, int nf_max,
                                            int upw, int sbp) {
  DecSmem s;
  size_t o = 0;
  s.xs2 = dec_take(o, (size_t)d * 4, 16);
  s.xg = dec_take(o, (size_t)(d / 64) * 4, 16);
  s.hs2 = dec_take(o, (size_t)k1 * I * 4, 16);
  s.hw = dec_take(o, (size_t)k1 * (I / 8) * 4, 16);
  s.gu = dec_take(o, (size_t)kDecWarps * upw * (d + d / 8), 128);
  s.dn = dec_take(o, (size_t)k1 * nf_max * (I / 2 + 4 * sbp), 128);
  s.rt = dec_take(o, (size_t)nf_max * Ep * 2, 128);
  s.outs = dec_take(o, (size_t)nf_max * 4, 16);
  s.lg = dec_take(o, (size_t)(E + 1) * 4, 16);
  s.sel_e = dec_take(o, kMaxK * 4, 16);
  s.sel_w = dec_take(o, kMaxK * 4, 16);
  s.misc = dec_take(o, 16, 16);
  s.red = dec_take(o, kDecWarps * 4, 16);
  s.bars = dec_take(o, (kDecWarps + 2) * 8, 8);
  s.ok = dec_take(o, 16, 16);
  s.total = o;
  return s;
}

__device__ __forceinline__ float bf16f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

template <int B>
__device__ __forceinline__ float code_plus128(uint32_t bytes) {
  return __uint_as_float(__byte_perm(bytes, 0x43000000u, 0x7044 | (B << 8)));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  const unsigned long long ua = *reinterpret_cast<unsigned long long*>(&a);
  const unsigned long long ub = *reinterpret_cast<unsigned long long*>(&b);
  const unsigned long long uc = *reinterpret_cast<unsigned long long*>(&c);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ua), "l"(ub), "l"(uc));
  return *reinterpret_cast<float2*>(&d);
}

// acc += sum over the 8 codes of w (K indices 8m..8m+7) of (128 + q) * x,
// x given as the pairs (x[8m+2b], x[8m+2b+1]), b = 0..3
__device__ __forceinline__ float2 dot8(uint32_t w, float2 x0, float2 x1, float2 x2, float2 x3,
                                       float2 acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  acc = ffma2(make_float2(code_plus128<0>(lo), code_plus128<0>(hi)), x0, acc);
  acc = ffma2(make_float2(code_plus128<1>(lo), code_plus128<1>(hi)), x1, acc);
  acc = ffma2(make_float2(code_plus128<2>(lo), code_plus128<2>(hi)), x2, acc);
  acc = ffma2(make_float2(code_plus128<3>(lo), code_plus128<3>(hi)), x3, acc);
  return acc;
}

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

__device__ __forceinline__ double softmax_term(float v, double m) {
  if (m == INFINITY) return v == INFINITY ? 1.0 : 0.0;
  if (m == -INFINITY) return 1.0;
  return exp((double)v - m);
}

// Grid-wide barrier number n (0-based): arrivals are counted monotonically, so
// barrier n completes at (n + 1) * gridDim.x.  Bounded: on time-out (or when
// another CTA gave up) every CTA leaves the kernel.
__device__ bool grid_sync(const DecParams& p, unsigned n, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
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
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__device__ __forceinline__ bool copy_wait(const DecParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_wait_bounded(bar, parity, p.abort_flag, kWaitNs)) return true;
  atomicOr(p.err, MOE_DEVERR_WAIT_TIMEOUT);
  atomicExch(p.abort_flag, 1);
  return false;
}

__device__ __forceinline__ void stamp(const DecParams& p, int l, int i) {
  if (p.tr_ns && blockIdx.x == 0 && threadIdx.x == 0)
    p.tr_ns[(long long)l * 4 + i] = (int64_t)globaltimer_ns();
}

__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int d = p.d, E = p.E, k = p.k, I = p.I, Ep = p.Ep;
  const int k1 = k + (p.has_shared ? 1 : 0);
  const int ng = d / 64;
  const int nwi = I / 8;  // words per down row
  const int sbp = p.sbp;
  const DecSmem L = dec_smem(d, I, k1, E, Ep, p.nf_max, p.upw, sbp);
  float2* xs2 = reinterpret_cast<float2*>(dsm + L.xs2);  // [32 pairs][ng]
  float* xg = reinterpret_cast<float*>(dsm + L.xg);      // [ng]
  float2* hs2 = reinterpret_cast<float2*>(dsm + L.hs2);  // [k1][4 pairs][I/8]
  float* hw = reinterpret_cast<float*>(dsm + L.hw);      // [k1][I/8]
  uint8_t* gu_buf = dsm + L.gu;
  uint8_t* dn_buf = dsm + L.dn;
  const uint16_t* rt_buf = reinterpret_cast<const uint16_t*>(dsm + L.rt);
  float* outs = reinterpret_cast<float*>(dsm + L.outs);
  float* lg = reinterpret_cast<float*>(dsm + L.lg);
  int* sel_e = reinterpret_cast<int*>(dsm + L.sel_e);
  float* sel_w = reinterpret_cast<float*>(dsm + L.sel_w);
  float* misc = reinterpret_cast<float*>(dsm + L.misc);  // [0] sigma, [1] 1/rms
  float* red = reinterpret_cast<float*>(dsm + L.red);
  const uint32_t bar0 = smem_u32(dsm + L.bars);  // [warps] gate/up, then down, router
  int* s_ok = reinterpret_cast<int*>(dsm + L.ok);
  const uint32_t dn_bar = bar0 + 8 * kDecWarps;
  const uint32_t rt_bar = bar0 + 8 * (kDecWarps + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int f0 = (int)((long long)c * d / G), f1 = (int)((long long)(c + 1) * d / G);
  const int nf = f1 - f0;
  const int U = k1 * I;
  const int u0 = (int)((long long)c * U / G), u1 = (int)((long long)(c + 1) * U / G);
  const int wu0 = min(u0 + warp * p.upw, u1);
  const int wu1 = min(wu0 + p.upw, u1);
  const int nu = wu1 - wu0;
  const int gu_unit = d + d / 8;
  const int dn_stride = p.nf_max * (I / 2 + 4 * sbp);

  if (tid == 0) {
    for (int i = 0; i < kDecWarps + 2; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t ph_gu = 0, ph_dn = 0, ph_rt = 0;
  unsigned nsync = 0;

  // x (bf16 [d]) -> shared memory in the lane-interleaved pair layout, with
  // optional RMS normalisation; also the owned features' values and the
  // group sums.  Returns 1/rms (1 when not normalised).
  auto load_x = [&](const uint16_t* src, bool norm, bool keep_own) -> float {
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
    float* xf = reinterpret_cast<float*>(xs2);
    for (int i = tid; i < d; i += kDecThreads) {
      const float v = bf16f(__ldcg(src + i)) * r;
      const int g = i >> 6, e = i & 63;
      xf[((e >> 1) * ng + g) * 2 + (e & 1)] = v;
      if (keep_own && i >= f0 && i < f1) outs[i - f0] = v;
    }
    __syncthreads();
    for (int g = warp; g < ng; g += kDecWarps) {
      const float2 v = xs2[lane * ng + g];
      const float s = warp_sum(v.x + v.y);
      if (lane == 0) xg[g] = s;
    }
    __syncthreads();
    return r;
  };

  // P_dst[e] += sum_{f owned} outs[f] * W'[e][f]  (e = E: the shared gate)
  auto router_partial = [&](unsigned long long* Pl) {
    for (int e = tid; e <= E; e += kDecThreads) {
      float acc = 0.f;
      for (int f = 0; f < nf; ++f) acc = fmaf(outs[f], bf16f(rt_buf[f * Ep + e]), acc);
      const long long v = __float2ll_rn(acc * kFix);
      atomicAdd(Pl + e, (unsigned long long)v);
    }
  };

  auto issue_router_copy = [&](int l) {
    if (tid == kDecThreads - 32 && nf > 0) {  // lane 0 of the last warp
      const uint32_t bytes = (uint32_t)nf * Ep * 2;
      mbar_arrive_expect_tx(rt_bar, bytes);
      bulk_g2s(smem_u32(dsm + L.rt), p.layer[l].w_rt + (long long)f0 * Ep, bytes, rt_bar);
    }
  };

  // ---- prologue: x_0 and the router sums of layer 0
  load_x(p.x, p.norm_first != 0, true);
  issue_router_copy(0);
  if (nf > 0) {
    if (!copy_wait(p, rt_bar, ph_rt)) return;
  }
  ph_rt ^= 1;
  if (nf > 0) router_partial(p.P);
  if (!grid_sync(p, nsync++, s_ok)) return;

  for (int l = 0; l < p.L; ++l) {
    const DecLayer& W = p.layer[l];
    stamp(p, l, 0);
    // ---- A: x_l, logits, top-k, copies
    const float r = (l == 0) ? 1.0f : load_x(p.out, true, false);
    for (int e = tid; e <= E; e += kDecThreads) {
      const long long s = (long long)__ldcg(p.P + (long long)l * (E + 1) + e);
      float v = (float)((double)s * (1.0 / 4294967296.0)) * r;
      if (e < E) {
        if (p.bias) v += p.bias[(long long)l * E + e];
        lg[e] = v;
        if (c == 0) p.logits[(long long)l * E + e] = v;
      } else {
        const float sg = p.has_shared ? 1.0f / (1.0f + expf(-v)) : 0.0f;
        misc[0] = sg;
        if (c == 0) p.sigma[l] = sg;
      }
    }
    __syncthreads();
    if (warp == 0) {
      constexpr int VPL = kMaxE / 32;
      uint32_t key[VPL];
      bool nan_seen = false;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        float v = -INFINITY;
        if (e < E) {
          v = lg[e];
          if (v != v) {
            v = -INFINITY;
            nan_seen = true;
          }
        }
        key[j] = (e < E) ? ord_key(v) : 0u;
      }
      if (__any_sync(0xffffffffu, nan_seen) && lane == 0 && c == 0)
        atomicOr(p.err, MOE_DEVERR_NAN_LOGIT);
      uint32_t taken = 0;
      for (int rr = 0; rr < k; ++rr) {
        uint32_t bk = 0;
        int be = INT_MAX;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int e = lane + 32 * j;
          if (e < E && !((taken >> j) & 1u) && (key[j] > bk || be == INT_MAX)) {
            bk = key[j];
            be = e;
          }
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t win = __reduce_min_sync(
            0xffffffffu, (bk == m && be != INT_MAX) ? (uint32_t)be : 0xFFFFFFFFu);
        if ((int)(win & 31) == lane) taken |= 1u << (win >> 5);
        if (lane == 0) sel_e[rr] = (int)win;
      }
      __syncwarp();
      const int my_e = (lane < k) ? sel_e[lane] : 0;
      float my_v = (lane < k) ? lg[my_e] : -INFINITY;
      if (my_v != my_v) my_v = -INFINITY;
      float top = lg[sel_e[0]];
      if (top != top) top = -INFINITY;
      const double m = (double)top;
      const double ex = (lane < k) ? softmax_term(my_v, m) : 0.0;
      double den = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      if (lane < k) {
        const float wv = (float)(ex / den);
        sel_w[lane] = wv;
        if (c == 0) {
          if (p.tr_idx) p.tr_idx[(long long)l * k + lane] = my_e;
          if (p.tr_w) p.tr_w[(long long)l * k + lane] = wv;
        }
      }
    }
    __syncthreads();
    // bulk copies: the warp's gate/up units, the CTA's down rows, the next router
    if (lane == 0 && nu > 0) {
      const uint32_t bar = bar0 + 8 * warp;
      mbar_arrive_expect_tx(bar, (uint32_t)(nu * gu_unit));
      for (int t = 0; t < nu; ++t) {
        const int u = wu0 + t;
        const int j = u / I, f = u - (u / I) * I;
        const long long ex = (j < k) ? sel_e[j] : E;
        const long long rg = ex * 2 * I + f, ru = rg + I;
        const uint32_t dst = smem_u32(gu_buf + (size_t)(warp * p.upw + t) * gu_unit);
        bulk_g2s(dst, W.gu_codes + rg * (d / 2), d / 2, bar);
        bulk_g2s(dst + d / 2, W.gu_codes + ru * (d / 2), d / 2, bar);
        bulk_g2s(dst + d, W.gu_sb + rg * ng, d / 16, bar);
        bulk_g2s(dst + d + d / 16, W.gu_sb + ru * ng, d / 16, bar);
      }
    }
    if (tid == 32 && nf > 0) {  // lane 0 of warp 1: the down rows of the k+1 experts
      mbar_arrive_expect_tx(dn_bar, (uint32_t)(k1 * nf * (I / 2 + 4 * sbp)));
      for (int j = 0; j < k1; ++j) {
        const long long ex = (j < k) ? sel_e[j] : E;
        const uint32_t dst = smem_u32(dn_buf + (size_t)j * dn_stride);
        bulk_g2s(dst, W.dn_codes + (ex * d + f0) * (I / 2), (uint32_t)nf * (I / 2), dn_bar);
        bulk_g2s(dst + p.nf_max * (I / 2), W.dn_sb + (ex * d + f0) * sbp, (uint32_t)nf * 4 * sbp,
                 dn_bar);
      }
    }
    if (l + 1 < p.L) issue_router_copy(l + 1);
    stamp(p, l, 1);

    // ---- GU: h = silu(gate . x) * (up . x) for the warp's units
    if (nu > 0) {
      if (!copy_wait(p, bar0 + 8 * warp, ph_gu)) return;
      float ag[kMaxUnitsPerWarp], au[kMaxUnitsPerWarp];
#pragma unroll
      for (int t = 0; t < kMaxUnitsPerWarp; ++t) ag[t] = au[t] = 0.f;
      for (int g = lane; g < ng; g += 32) {
        float2 xv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[i] = xs2[i * ng + g];
        const float X = xg[g];
#pragma unroll
        for (int t = 0; t < kMaxUnitsPerWarp; ++t) {
          if (t < nu) {
            const uint8_t* ub = gu_buf + (size_t)(warp * p.upw + t) * gu_unit;
            const uint4 cg0 = *reinterpret_cast<const uint4*>(ub + g * 32);
            const uint4 cg1 = *reinterpret_cast<const uint4*>(ub + g * 32 + 16);
            const uint4 cu0 = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32);
            const uint4 cu1 = *reinterpret_cast<const uint4*>(ub + d / 2 + g * 32 + 16);
            const uint32_t sbg = reinterpret_cast<const uint32_t*>(ub + d)[g];
            const uint32_t sbu = reinterpret_cast<const uint32_t*>(ub + d + d / 16)[g];
            float2 pg = make_float2(0.f, 0.f), pu = make_float2(0.f, 0.f);
            pg = dot8(cg0.x, xv[0], xv[1], xv[2], xv[3], pg);
            pu = dot8(cu0.x, xv[0], xv[1], xv[2], xv[3], pu);
            pg = dot8(cg0.y, xv[4], xv[5], xv[6], xv[7], pg);
            pu = dot8(cu0.y, xv[4], xv[5], xv[6], xv[7], pu);
            pg = dot8(cg0.z, xv[8], xv[9], xv[10], xv[11], pg);
            pu = dot8(cu0.z, xv[8], xv[9], xv[10], xv[11], pu);
            pg = dot8(cg0.w, xv[12], xv[13], xv[14], xv[15], pg);
            pu = dot8(cu0.w, xv[12], xv[13], xv[14], xv[15], pu);
            pg = dot8(cg1.x, xv[16], xv[17], xv[18], xv[19], pg);
            pu = dot8(cu1.x, xv[16], xv[17], xv[18], xv[19], pu);
            pg = dot8(cg1.y, xv[20], xv[21], xv[22], xv[23], pg);
            pu = dot8(cu1.y, xv[20], xv[21], xv[22], xv[23], pu);
            pg = dot8(cg1.z, xv[24], xv[25], xv[26], xv[27], pg);
            pu = dot8(cu1.z, xv[24], xv[25], xv[26], xv[27], pu);
            pg = dot8(cg1.w, xv[28], xv[29], xv[30], xv[31], pg);
            pu = dot8(cu1.w, xv[28], xv[29], xv[30], xv[31], pu);
            ag[t] += s_of(sbg) * ((pg.x + pg.y) - 128.0f * X) + b_of(sbg) * X;
            au[t] += s_of(sbu) * ((pu.x + pu.y) - 128.0f * X) + b_of(sbu) * X;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kMaxUnitsPerWarp; ++t) {
        if (t < nu) {
          const float g = warp_sum(ag[t]);
          const float u = warp_sum(au[t]);
          if (lane == 0) p.H[wu0 + t] = g / (1.0f + expf(-g)) * u;  // unit = j*I + f
        }
      }
    }
    ph_gu ^= 1;
    if (!grid_sync(p, nsync++, s_ok)) return;
    stamp(p, l, 2);

    // ---- D: h of every active expert -> shared memory (pair layout + word sums)
    {
      float* hf = reinterpret_cast<float*>(hs2);
      for (int i = tid; i < k1 * I; i += kDecThreads) {
        const int j = i / I, e = i - j * I;
        const int w = e >> 3, q = (e & 7) >> 1;
        hf[(((j * 4 + q) * nwi) + w) * 2 + (e & 1)] = __ldcg(p.H + i);
      }
      __syncthreads();
      for (int i = tid; i < k1 * nwi; i += kDecThreads) {
        const int j = i / nwi, w = i - j * nwi;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 v = hs2[(j * 4 + q) * nwi + w];
          s += v.x + v.y;
        }
        hw[i] = s;
      }
      __syncthreads();
    }
    if (nf > 0) {
      if (!copy_wait(p, dn_bar, ph_dn)) return;
    }
    ph_dn ^= 1;
    {
      const float sigma = misc[0];
      for (int fl = warp; fl < nf; fl += kDecWarps) {
        float outv = 0.f;
        for (int j = 0; j < k1; ++j) {
          const uint8_t* rowc = dn_buf + (size_t)j * dn_stride + (size_t)fl * (I / 2);
          const uint32_t* rows = reinterpret_cast<const uint32_t*>(
              dn_buf + (size_t)j * dn_stride + (size_t)p.nf_max * (I / 2) + (size_t)fl * 4 * sbp);
          float a = 0.f;
          for (int w = lane; w < nwi; w += 32) {
            const uint32_t cw = reinterpret_cast<const uint32_t*>(rowc)[w];
            const float2* hp = hs2 + (size_t)j * 4 * nwi + w;
            const float2 acc =
                dot8(cw, hp[0], hp[nwi], hp[2 * nwi], hp[3 * nwi], make_float2(0.f, 0.f));
            const float Hs = hw[j * nwi + w];
            const uint32_t sb = rows[w >> 3];
            a += s_of(sb) * ((acc.x + acc.y) - 128.0f * Hs) + b_of(sb) * Hs;
          }
          a = warp_sum(a);
          outv += ((j < k) ? sel_w[j] : sigma) * a;
        }
        if (lane == 0) {
          const uint16_t o = __bfloat16_as_ushort(__float2bfloat16_rn(outv));
          const int f = f0 + fl;
          outs[fl] = bf16f(o);
          p.out[f] = o;
          if (p.tr_out) p.tr_out[(long long)l * d + f] = o;
          if (l == p.L - 1) p.y[f] = o;
        }
      }
    }
    __syncthreads();
    stamp(p, l, 3);
    if (l + 1 < p.L) {
      if (nf > 0) {
        if (!copy_wait(p, rt_bar, ph_rt)) return;
      }
      ph_rt ^= 1;
      if (nf > 0) router_partial(p.P + (long long)(l + 1) * (E + 1));
      if (!grid_sync(p, nsync++, s_ok)) return;
    }
  }
}

}  // namespace

size_t decode_scratch_bytes(const Handle* h, int L) {
  const moe_config& c = h->cfg;
  return 256 + (size_t)L * c.E * 4 + (size_t)L * 4 + (size_t)(c.k + 1) * c.I * 4 + (size_t)c.d * 2 +
         (size_t)L * (c.E + 1) * 8 + 2048;
}

cudaError_t launch_decode(Handle* const* layers, int L, const uint16_t* x, const float* bias,
                          float eps, uint16_t* y, const moe_decode_trace* trace,
                          cudaStream_t st) {
  const Handle* h0 = layers[0];
  const moe_config& c = h0->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const int G = h0->num_sms;
  const int nf_max = (c.d + G - 1) / G;
  const int units_cta = (k1 * c.I + G - 1) / G;
  const int upw = (units_cta + kDecWarps - 1) / kDecWarps;
  if (upw > kMaxUnitsPerWarp) return cudaErrorInvalidConfiguration;
  const int Ep = decode_router_pitch(c.E);
  const int sbp = decode_dn_sb_pitch(c.I);
  const DecSmem sm = dec_smem(c.d, c.I, k1, c.E, Ep, nf_max, upw, sbp);
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
  for (int l0 = 0; l0 < L; l0 += kMaxDecLayers) {
    const int nl = (L - l0) < kMaxDecLayers ? (L - l0) : kMaxDecLayers;
    DecParams p;
    for (int i = 0; i < nl; ++i) {
      const Handle* h = layers[l0 + i];
      const long long gu_codes = (long long)h->n_exp * 2 * c.I * (c.d / 2);
      const long long dn_codes = (long long)h->n_exp * c.d * (c.I / 2);
      p.layer[i].gu_codes = h->dc_gu;
      p.layer[i].gu_sb = reinterpret_cast<const uint32_t*>(h->dc_gu + gu_codes);
      p.layer[i].dn_codes = h->dc_dn;
      p.layer[i].dn_sb = reinterpret_cast<const uint32_t*>(h->dc_dn + dn_codes);
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
    p.upw = upw;
    p.sbp = sbp;
    p.x = (l0 == 0) ? x : y;
    p.norm_first = (l0 == 0) ? 0 : 1;
    p.bias = bias ? bias + (long long)l0 * c.E : nullptr;
    p.eps = eps;
    p.y = y;
    uint8_t* q = scr;
    p.bar = reinterpret_cast<unsigned*>(q);
    p.abort_flag = reinterpret_cast<int*>(q + 4);
    q += 256;
    p.P = reinterpret_cast<unsigned long long*>(q);
    const size_t pbytes = (size_t)nl * (c.E + 1) * 8;
    q += (pbytes + 255) / 256 * 256;
    p.logits = (trace && trace->logits) ? trace->logits + (long long)l0 * c.E
                                        : reinterpret_cast<float*>(q);
    q += (size_t)kMaxDecLayers * c.E * 4;
    p.sigma = (trace && trace->sigma) ? trace->sigma + l0 : reinterpret_cast<float*>(q);
    q += (size_t)kMaxDecLayers * 4 + 256;
    p.H = reinterpret_cast<float*>(q);
    q += (size_t)k1 * c.I * 4 + 256;
    p.out = reinterpret_cast<uint16_t*>(q);
    p.tr_idx = (trace && trace->idx) ? trace->idx + (long long)l0 * c.k : nullptr;
    p.tr_w = (trace && trace->w) ? trace->w + (long long)l0 * c.k : nullptr;
    p.tr_out = (trace && trace->out)
                   ? reinterpret_cast<uint16_t*>(trace->out) + (long long)l0 * c.d
                   : nullptr;
    p.tr_ns = (trace && trace->timestamps) ? trace->timestamps + (long long)l0 * 4 : nullptr;
    p.err = h0->dev_err;
    // the barrier counter, the abort flag and the fixed-point sums start at zero
    cudaError_t e = cudaMemsetAsync(scr, 0, 256 + pbytes, st);
    if (e != cudaSuccess) return e;
    void* args[] = {&p};
    e = cudaLaunchCooperativeKernel((const void*)decode_kernel, dim3(G), dim3(kDecThreads), args,
                                    sm.total, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
