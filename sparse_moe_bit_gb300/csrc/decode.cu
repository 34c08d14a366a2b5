// Batch-1 decode path: one persistent cooperative kernel runs every layer of
// the chain on CUDA cores.  The work is bound by weight reads (4.5 bits per
// weight), so each phase spreads its rows over all SMs, streams the codes
// with 16-byte non-caching loads and reduces within a warp.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Optimizing the one-row weight path" (a row-parallel GEMV where a SIMD
// group cooperates on one output while reading different parts of the
// weight matrix), §"Reduce intermediate and state traffic" (gate and up
// projections fused with their gated activation; the output projection fused
// with its routing score and the shared expert's result) and §"Keep each
// decode step on the GPU" (no host synchronisation between the steps).
//
// Per layer l (x_l fp32 in shared memory of every CTA):
//   R : router logits and the shared-expert gate, one warp per expert row
//       -> grid barrier
//   GU: every CTA repeats the top-k selection from the logits; the
//       (expert, feature) units of the k + 1 active experts are split evenly
//       over the CTAs; one warp computes the gate and the up row of a unit and
//       h = silu(g) * u
//       -> grid barrier
//   D : every CTA owns a contiguous range of output features and computes,
//       for each, the k + 1 down rows and the weighted sum in fixed order
//       (slots 0..k-1, then the shared expert) -> out_l bf16
//       -> grid barrier; x_{l+1} = out_l / sqrt(mean(out_l^2) + eps)
// Dot products use the split s*q + beta: sum_i (s q_i + beta) x_i =
// s * sum_i q_i x_i + beta * sum_i x_i per 64-group, with the codes turned
// into floats by a byte permute into the fp32 pattern of 128 + q.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxDecLayers = 64;
constexpr uint64_t kGridWaitNs = 2000000000ull;

struct DecLayer {
  const uint8_t* gu_codes;  // [n_exp][2I][d/2]
  const uint32_t* gu_sb;    // [n_exp][2I][d/64]
  const uint8_t* dn_codes;  // [n_exp][d][I/2]
  const uint32_t* dn_sb;    // [n_exp][d][I/64]
  const uint16_t* w_router; // bf16 [E][d]
  const uint16_t* w_sg;     // bf16 [d]
};

struct DecParams {
  DecLayer layer[kMaxDecLayers];
  int L, d, E, k, I, has_shared;
  const uint16_t* x;
  int norm_first;     // 1: x is a previous layer's output (normalise it first)
  const float* bias;  // [L][E] or null
  float eps;
  uint16_t* y;
  float* logits;      // [L][E]
  float* sigma;       // [L]
  int32_t* tr_idx;    // [L][k] or null
  float* tr_w;        // [L][k] or null
  uint16_t* tr_out;   // [L][d] or null
  float* H;           // [(k+1)][I]
  uint16_t* out;      // [d]
  unsigned* bar;      // grid barrier arrivals (zero at launch)
  int* abort_flag;    // zero at launch
  int* err;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// float value 128 + q of the code in byte `b` (0..3) of a word whose bytes
// each hold one code in their low nibble
template <int B>
__device__ __forceinline__ float code_plus128(uint32_t bytes) {
  return __uint_as_float(__byte_perm(bytes, 0x43000000u, 0x7044 | (B << 8)));
}

// sum over 8 codes of word w (K indices 8m..8m+7) of (128 + q_i) * x_i
__device__ __forceinline__ float dot8(uint32_t w, const float* x, float acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // K indices 8m, 8m+2, 8m+4, 8m+6
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // K indices 8m+1, 8m+3, ...
  acc = fmaf(code_plus128<0>(lo), x[0], acc);
  acc = fmaf(code_plus128<0>(hi), x[1], acc);
  acc = fmaf(code_plus128<1>(lo), x[2], acc);
  acc = fmaf(code_plus128<1>(hi), x[3], acc);
  acc = fmaf(code_plus128<2>(lo), x[4], acc);
  acc = fmaf(code_plus128<2>(hi), x[5], acc);
  acc = fmaf(code_plus128<3>(lo), x[6], acc);
  acc = fmaf(code_plus128<3>(hi), x[7], acc);
  return acc;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Grid-wide barrier number `n` (0-based): arrivals are counted monotonically,
// so barrier n completes at (n + 1) * gridDim.x.  The wait is bounded; on
// time-out (or if another CTA gave up) every CTA leaves the kernel.
__device__ bool grid_sync(const DecParams& p, unsigned n, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(p.bar, 1u);
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
        if (globaltimer_ns() - t0 > kGridWaitNs) {
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

__device__ __forceinline__ bool beats(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ float dsm[];
  const int d = p.d, E = p.E, k = p.k, I = p.I;
  const int k1 = k + (p.has_shared ? 1 : 0);
  const int ng = d / 64;  // groups along d
  float* xs = dsm;              // [d]
  float* xg = xs + d;           // [d/64] group sums of x
  float* hs = xg + ng;          // [k1][I]
  float* hg = hs + k1 * I;      // [k1][I/16] sums of 16 consecutive h
  int* sel_e = reinterpret_cast<int*>(hg + k1 * (I / 16));  // [k]
  float* sel_w = reinterpret_cast<float*>(sel_e + kMaxK);   // [k]
  float* misc = sel_w + kMaxK;                                // [0] sigma, [1] rms
  float* red = misc + 4;                                      // [kDecWarps]
  int* s_ok = reinterpret_cast<int*>(red + kDecWarps);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  unsigned nsync = 0;

  for (int l = 0; l < p.L; ++l) {
    const DecLayer& W = p.layer[l];
    // ---- x_l into shared memory (fp32), and its group sums
    if (l == 0 && !p.norm_first) {
      for (int c = threadIdx.x; c < d; c += kDecThreads)
        xs[c] = __uint_as_float((uint32_t)p.x[c] << 16);
    } else {
      // out_{l-1} was written by all CTAs before the last barrier
      const uint16_t* src = (l == 0) ? p.x : p.out;
      float ss = 0.f;
      for (int c = threadIdx.x; c < d; c += kDecThreads) {
        const float v = __uint_as_float((uint32_t)__ldcg(src + c) << 16);
        xs[c] = v;
        ss += v * v;
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < kDecWarps; ++w) t += red[w];
        misc[1] = rsqrtf(t / (float)d + p.eps);
      }
      __syncthreads();
      const float r = misc[1];
      for (int c = threadIdx.x; c < d; c += kDecThreads) xs[c] *= r;
    }
    __syncthreads();
    for (int g = warp; g < ng; g += kDecWarps) {
      float s = xs[g * 64 + lane] + xs[g * 64 + 32 + lane];
      s = warp_sum(s);
      if (lane == 0) xg[g] = s;
    }
    __syncthreads();

    // ---- R: router logits (+ shared gate), one warp per row
    {
      const int nrows = E + (p.has_shared ? 1 : 0);
      for (int e = blockIdx.x * kDecWarps + warp; e < nrows; e += G * kDecWarps) {
        const uint16_t* row = (e < E) ? W.w_router + (long long)e * d : W.w_sg;
        float acc = 0.f;
        for (int c = lane * 8; c < d; c += 256) {
          const uint4 v = ldg_stream(row + c);
          const float* xc = xs + c;
          acc = fmaf(bf16_lo(v.x), xc[0], acc);
          acc = fmaf(bf16_hi(v.x), xc[1], acc);
          acc = fmaf(bf16_lo(v.y), xc[2], acc);
          acc = fmaf(bf16_hi(v.y), xc[3], acc);
          acc = fmaf(bf16_lo(v.z), xc[4], acc);
          acc = fmaf(bf16_hi(v.z), xc[5], acc);
          acc = fmaf(bf16_lo(v.w), xc[6], acc);
          acc = fmaf(bf16_hi(v.w), xc[7], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) {
          if (e < E) {
            float v = acc;
            if (p.bias) v += p.bias[(long long)l * E + e];
            p.logits[(long long)l * E + e] = v;
          } else {
            p.sigma[l] = 1.0f / (1.0f + expf(-acc));
          }
        }
      }
    }
    if (!grid_sync(p, nsync++, s_ok)) return;

    // ---- top-k (every CTA, warp 0), fp64 weights
    if (warp == 0) {
      constexpr int VPL = kMaxE / 32;
      float v[VPL];
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        float s = -INFINITY;
        if (e < E) {
          s = __ldcg(p.logits + (long long)l * E + e);
          if (s != s) {
            s = -INFINITY;
            atomicOr(p.err, MOE_DEVERR_NAN_LOGIT);
          }
        }
        v[j] = s;
      }
      uint32_t taken = 0;
      for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int be = INT_MAX;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int e = lane + 32 * j;
          if (e < E && !((taken >> j) & 1u) && beats(v[j], e, bv, be)) {
            bv = v[j];
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (beats(ov, oe, bv, be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) {
          sel_e[r] = be;
          sel_w[r] = bv;  // logit for now
        }
      }
      __syncwarp();
      if (lane == 0) {
        const double m = (double)sel_w[0];
        double ex[kMaxK];
        double den = 0.0;
        for (int r = 0; r < k; ++r) {
          // softmax limit for infinite logits (as in the prefill top-k)
          if (m == INFINITY) ex[r] = (sel_w[r] == INFINITY) ? 1.0 : 0.0;
          else if (m == -INFINITY) ex[r] = 1.0;
          else ex[r] = exp((double)sel_w[r] - m);
          den += ex[r];
        }
        for (int r = 0; r < k; ++r) sel_w[r] = (float)(ex[r] / den);
        misc[0] = p.has_shared ? __ldcg(p.sigma + l) : 0.f;
        if (blockIdx.x == 0) {
          for (int r = 0; r < k; ++r) {
            if (p.tr_idx) p.tr_idx[(long long)l * k + r] = sel_e[r];
            if (p.tr_w) p.tr_w[(long long)l * k + r] = sel_w[r];
          }
        }
      }
    }
    __syncthreads();

    // ---- GU: units (slot j, feature f); gate row f and up row f of expert e_j
    {
      const int U = k1 * I;
      const int u0 = (int)((long long)blockIdx.x * U / G);
      const int u1 = (int)((long long)(blockIdx.x + 1) * U / G);
      for (int u = u0 + warp; u < u1; u += kDecWarps) {
        const int j = u / I;
        const int f = u - j * I;
        const int ex = (j < k) ? sel_e[j] : E;
        const long long rg = (long long)ex * 2 * I + f;
        const long long ru = rg + I;
        float ag = 0.f, au = 0.f;
        for (int g = lane; g < ng; g += 32) {
          const uint4 cg0 = ldg_stream(W.gu_codes + rg * (d / 2) + g * 32);
          const uint4 cg1 = ldg_stream(W.gu_codes + rg * (d / 2) + g * 32 + 16);
          const uint4 cu0 = ldg_stream(W.gu_codes + ru * (d / 2) + g * 32);
          const uint4 cu1 = ldg_stream(W.gu_codes + ru * (d / 2) + g * 32 + 16);
          const uint32_t sbg = __ldg(W.gu_sb + rg * ng + g);
          const uint32_t sbu = __ldg(W.gu_sb + ru * ng + g);
          const float* xc = xs + g * 64;
          float pg = 0.f, pu = 0.f;
          pg = dot8(cg0.x, xc + 0, pg);
          pu = dot8(cu0.x, xc + 0, pu);
          pg = dot8(cg0.y, xc + 8, pg);
          pu = dot8(cu0.y, xc + 8, pu);
          pg = dot8(cg0.z, xc + 16, pg);
          pu = dot8(cu0.z, xc + 16, pu);
          pg = dot8(cg0.w, xc + 24, pg);
          pu = dot8(cu0.w, xc + 24, pu);
          pg = dot8(cg1.x, xc + 32, pg);
          pu = dot8(cu1.x, xc + 32, pu);
          pg = dot8(cg1.y, xc + 40, pg);
          pu = dot8(cu1.y, xc + 40, pu);
          pg = dot8(cg1.z, xc + 48, pg);
          pu = dot8(cu1.z, xc + 48, pu);
          pg = dot8(cg1.w, xc + 56, pg);
          pu = dot8(cu1.w, xc + 56, pu);
          const float X = xg[g];
          const float sg = __half2float(__ushort_as_half((uint16_t)(sbg & 0xFFFFu)));
          const float bg = __half2float(__ushort_as_half((uint16_t)(sbg >> 16)));
          const float su = __half2float(__ushort_as_half((uint16_t)(sbu & 0xFFFFu)));
          const float bu = __half2float(__ushort_as_half((uint16_t)(sbu >> 16)));
          ag += sg * (pg - 128.0f * X) + bg * X;
          au += su * (pu - 128.0f * X) + bu * X;
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) p.H[(long long)j * I + f] = ag / (1.0f + expf(-ag)) * au;
      }
    }
    if (!grid_sync(p, nsync++, s_ok)) return;

    // ---- D: h into shared memory, then the owned output features
    for (int i = threadIdx.x; i < k1 * I; i += kDecThreads) hs[i] = __ldcg(p.H + i);
    __syncthreads();
    for (int i = threadIdx.x; i < k1 * (I / 16); i += kDecThreads) {
      float s = 0.f;
      for (int q = 0; q < 16; ++q) s += hs[i * 16 + q];
      hg[i] = s;
    }
    __syncthreads();
    {
      const int f0 = (int)((long long)blockIdx.x * d / G);
      const int f1 = (int)((long long)(blockIdx.x + 1) * d / G);
      const int ngi = I / 64;
      const float sigma = misc[0];
      for (int f = f0 + warp; f < f1; f += kDecWarps) {
        float outv = 0.f;
        for (int j = 0; j < k1; ++j) {
          const int ex = (j < k) ? sel_e[j] : E;
          const long long row = (long long)ex * d + f;
          float a = 0.f;
          for (int i = lane * 16; i < I; i += 512) {
            const uint2 c = ldg_stream2(W.dn_codes + row * (I / 2) + i / 2);
            const uint32_t sb = __ldg(W.dn_sb + row * ngi + i / 64);
            const float* hc = hs + j * I + i;
            float acc = dot8(c.x, hc, 0.f);
            acc = dot8(c.y, hc + 8, acc);
            const float Hsum = hg[j * (I / 16) + i / 16];
            const float s = __half2float(__ushort_as_half((uint16_t)(sb & 0xFFFFu)));
            const float b = __half2float(__ushort_as_half((uint16_t)(sb >> 16)));
            a += s * (acc - 128.0f * Hsum) + b * Hsum;
          }
          a = warp_sum(a);
          outv += ((j < k) ? sel_w[j] : sigma) * a;
        }
        if (lane == 0) {
          const uint16_t o = __bfloat16_as_ushort(__float2bfloat16_rn(outv));
          p.out[f] = o;
          if (p.tr_out) p.tr_out[(long long)l * d + f] = o;
          if (l == p.L - 1) p.y[f] = o;
        }
      }
    }
    if (l + 1 < p.L) {
      if (!grid_sync(p, nsync++, s_ok)) return;
    }
  }
}

}  // namespace

size_t decode_scratch_bytes(const Handle* h, int L) {
  const moe_config& c = h->cfg;
  return (size_t)L * c.E * 4 + (size_t)L * 4 + (size_t)(c.k + 1) * c.I * 4 + (size_t)c.d * 2 +
         256;
}

cudaError_t launch_decode(Handle* const* layers, int L, const uint16_t* x, const float* bias,
                          float eps, uint16_t* y, const moe_decode_trace* trace,
                          cudaStream_t st) {
  const Handle* h0 = layers[0];
  const moe_config& c = h0->cfg;
  // scratch lives in the first layer's workspace area reserved for decode
  uint8_t* scr = reinterpret_cast<uint8_t*>(h0->ws.logit_part);
  static_assert(sizeof(DecParams) < 32000, "kernel parameter size");
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
      p.layer[i].w_router = h->w_router;
      p.layer[i].w_sg = h->w_sg;
    }
    p.L = nl;
    p.d = c.d;
    p.E = c.E;
    p.k = c.k;
    p.I = c.I;
    p.has_shared = c.has_shared;
    p.x = x;
    p.norm_first = 0;
    p.bias = bias ? bias + (long long)l0 * c.E : nullptr;
    p.eps = eps;
    p.y = y;
    // scratch carve-up
    uint8_t* q = scr;
    unsigned* bar = reinterpret_cast<unsigned*>(q);
    int* abort_flag = reinterpret_cast<int*>(q + 4);
    q += 256;
    p.logits = (trace && trace->logits) ? trace->logits + (long long)l0 * c.E
                                        : reinterpret_cast<float*>(q);
    q += (size_t)kMaxDecLayers * c.E * 4;
    p.sigma = (trace && trace->sigma) ? trace->sigma + l0 : reinterpret_cast<float*>(q);
    q += (size_t)kMaxDecLayers * 4;
    p.H = reinterpret_cast<float*>(q);
    q += (size_t)(c.k + 1) * c.I * 4;
    p.out = reinterpret_cast<uint16_t*>(q);
    p.tr_idx = (trace && trace->idx) ? trace->idx + (long long)l0 * c.k : nullptr;
    p.tr_w = (trace && trace->w) ? trace->w + (long long)l0 * c.k : nullptr;
    p.tr_out = (trace && trace->out)
                   ? reinterpret_cast<uint16_t*>(trace->out) + (long long)l0 * c.d
                   : nullptr;
    p.bar = bar;
    p.abort_flag = abort_flag;
    p.err = h0->dev_err;
    // a later group starts from the previous group's output
    if (l0 > 0) {
      p.x = y;
      p.norm_first = 1;
    }

    cudaError_t e = cudaMemsetAsync(bar, 0, 8, st);
    if (e != cudaSuccess) return e;
    const int k1 = c.k + (c.has_shared ? 1 : 0);
    const size_t smem = (size_t)(c.d + c.d / 64 + k1 * c.I + k1 * (c.I / 16)) * 4 +
                        2 * kMaxK * 4 + 16 + kDecWarps * 4 + 16;
    static bool attr = false;
    if (!attr) {
      e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    void* args[] = {&p};
    e = cudaLaunchCooperativeKernel((const void*)decode_kernel, dim3(h0->num_sms),
                                    dim3(kDecThreads), args, smem, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
