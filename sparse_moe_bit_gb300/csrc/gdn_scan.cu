// Gated DeltaNet prefill scan with the recurrent state held in registers.
//
// Operation (Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Qwen creates three different workload shapes" and §"Keep recurrent state
// on chip"): each value head carries a state matrix S [dv x dk] through the
// prompt; per token a gate alpha = exp(g) keeps part of it and a delta update
// of strength beta writes the token's value under its key (the gated delta
// rule):
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
//     o_t = scale S_t q_t
// State and gate in fp32, q, k, v in bf16, o rounded to bf16.  Value head h
// reads query/key head h / (Hv / Hk).
//
// Design.  Row i of S evolves on its own:
//     u      = S_{t-1}[i] . k_t
//     c      = beta_t (v_t[i] - alpha_t u)
//     S_t[i] = alpha_t S_{t-1}[i] + c k_t
//     o_t[i] = alpha_t (S_{t-1}[i] . q~_t) + c (k_t . q~_t),   q~ = scale q
// (the readout from the identity S_t q = alpha S_{t-1} q + c (k . q), so one
// pass over the row per token serves both dot products).  Eight lanes share
// one row, 16 fp32 state values each, for the whole scan: the state never
// leaves registers until the end.  The two dot products are summed across
// the eight lanes by a shuffle butterfly, after which all eight hold the same
// c (addition is commutative, so the butterfly gives every lane identical
// bits).  A CTA of 256 threads holds 32 rows of one head; grid (dv/32, Hv,
// sequences).  Tokens are staged 32 at a time in shared memory as fp32
// (k and scaled q, the 32 rows' v values, alpha, beta and k . q~ per token),
// double-buffered: the next block's global loads are issued into registers
// before the current block is scanned and stored to the other buffer after.
// Lane s of a row holds columns 32 m + 4 s + e (m, e < 4), so the eight
// distinct float4 addresses one warp reads per load cover all 32 banks.
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kDk = kGdnDk;             // state columns (key width)
constexpr int kRows = kGdnRows;         // state rows per CTA
constexpr int kLanes = 8;               // lanes per row
constexpr int kThreads = kRows * kLanes;  // 256
constexpr int kChunk = 32;              // tokens per staged block
constexpr int kVec = kDk / (4 * kLanes);  // float4 groups per lane (4)

static_assert(kThreads == 256 && kVec == 4, "layout below assumes these");
static_assert(kChunk * kDk / 8 == 2 * kThreads, "two 16-byte loads of k (and q) per thread");
static_assert(kChunk * kRows / 8 == kThreads / 2, "one 16-byte load of v per thread of the first half");

struct __align__(16) GdnSmem {
  float k[2][kChunk][kDk];
  float q[2][kChunk][kDk];       // scaled by the readout scale
  float v[2][kChunk][kRows];
  float4 sc[2][kChunk];          // alpha, beta, k . q~, unused
  float o[kChunk][kRows];
};

// One staged block, in flight in registers.
struct Prefetch {
  uint4 k[2], q[2], v;
  float gb;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  // round to nearest even (finite values)
  uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  ua = (ua + 0x7FFFu + ((ua >> 16) & 1u)) >> 16;
  ub = (ub + 0x7FFFu + ((ub >> 16) & 1u)) >> 16;
  return ua | (ub << 16);
}

// Issue the global loads of tokens t0 .. t0+n-1 (n <= kChunk; lanes past n
// load nothing and hold zeros).
__device__ __forceinline__ void load_block(Prefetch& pf, const GdnParams& p, int h, int hk,
                                           int r0, int t0, int n, int tid) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + j * kThreads;          // 16-byte piece of the block's k (q)
    const int tt = i >> 4, c8 = (i & 15) * 8;  // token, first column
    pf.k[j] = make_uint4(0, 0, 0, 0);
    pf.q[j] = make_uint4(0, 0, 0, 0);
    if (tt < n) {
      const size_t off = ((size_t)(t0 + tt) * p.Hk + hk) * kDk + c8;
      pf.k[j] = __ldg(reinterpret_cast<const uint4*>(p.k + off));
      pf.q[j] = __ldg(reinterpret_cast<const uint4*>(p.q + off));
    }
  }
  pf.v = make_uint4(0, 0, 0, 0);
  pf.gb = 0.f;
  if (tid < kThreads / 2) {
    const int tt = tid >> 2, c8 = (tid & 3) * 8;
    if (tt < n)
      pf.v = __ldg(reinterpret_cast<const uint4*>(p.v + ((size_t)(t0 + tt) * p.Hv + h) * p.dv +
                                                  r0 + c8));
  } else if (tid < kThreads / 2 + 2 * kChunk) {
    const int tt = (tid - kThreads / 2) & (kChunk - 1);
    const bool is_beta = tid >= kThreads / 2 + kChunk;
    if (tt < n) {
      const size_t off = (size_t)(t0 + tt) * p.Hv + h;
      pf.gb = is_beta ? __ldg(p.beta + off) : __ldg(p.g + off);
    }
  }
}

__device__ __forceinline__ void store_block(GdnSmem& sm, int b, const Prefetch& pf, float scale,
                                            int tid) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + j * kThreads;
    const int tt = i >> 4, c8 = (i & 15) * 8;
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(&pf.k[j]);
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(&pf.q[j]);
    float4* kd = reinterpret_cast<float4*>(&sm.k[b][tt][c8]);
    float4* qd = reinterpret_cast<float4*>(&sm.q[b][tt][c8]);
    kd[0] = make_float4(bf16_lo(kw[0]), bf16_hi(kw[0]), bf16_lo(kw[1]), bf16_hi(kw[1]));
    kd[1] = make_float4(bf16_lo(kw[2]), bf16_hi(kw[2]), bf16_lo(kw[3]), bf16_hi(kw[3]));
    qd[0] = make_float4(scale * bf16_lo(qw[0]), scale * bf16_hi(qw[0]), scale * bf16_lo(qw[1]),
                        scale * bf16_hi(qw[1]));
    qd[1] = make_float4(scale * bf16_lo(qw[2]), scale * bf16_hi(qw[2]), scale * bf16_lo(qw[3]),
                        scale * bf16_hi(qw[3]));
  }
  if (tid < kThreads / 2) {
    const int tt = tid >> 2, c8 = (tid & 3) * 8;
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(&pf.v);
    float4* vd = reinterpret_cast<float4*>(&sm.v[b][tt][c8]);
    vd[0] = make_float4(bf16_lo(vw[0]), bf16_hi(vw[0]), bf16_lo(vw[1]), bf16_hi(vw[1]));
    vd[1] = make_float4(bf16_lo(vw[2]), bf16_hi(vw[2]), bf16_lo(vw[3]), bf16_hi(vw[3]));
  } else if (tid < kThreads / 2 + kChunk) {
    sm.sc[b][tid - kThreads / 2].x = expf(pf.gb);        // alpha, fp32
  } else if (tid < kThreads / 2 + 2 * kChunk) {
    sm.sc[b][tid - kThreads / 2 - kChunk].y = pf.gb;     // beta
  }
}

// k . q~ of each staged token: eight threads per token, same column split as
// the state rows.
__device__ __forceinline__ void block_kq(GdnSmem& sm, int b, int tid) {
  const int tt = tid >> 3, s = tid & 7;
  float acc = 0.f;
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    const float4 a = *reinterpret_cast<const float4*>(&sm.k[b][tt][32 * m + 4 * s]);
    const float4 c = *reinterpret_cast<const float4*>(&sm.q[b][tt][32 * m + 4 * s]);
    acc = fmaf(a.x, c.x, acc);
    acc = fmaf(a.y, c.y, acc);
    acc = fmaf(a.z, c.z, acc);
    acc = fmaf(a.w, c.w, acc);
  }
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
  if (s == 0) sm.sc[b][tt].z = acc;
}

__global__ void __launch_bounds__(kThreads, 1) gdn_scan_kernel(const GdnParams p) {
  extern __shared__ float4 gdn_smem_raw[];
  GdnSmem& sm = *reinterpret_cast<GdnSmem*>(gdn_smem_raw);
  const int tid = threadIdx.x;
  const int row = tid >> 3, s = tid & 7;
  const int r0 = blockIdx.x * kRows, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);

  int beg = 0, end = p.T;
  if (p.offsets) {
    beg = min(max(__ldg(p.offsets + n), 0), p.T);
    end = min(max(__ldg(p.offsets + n + 1), beg), p.T);
  }

  // The row's 16 state values: columns 32 m + 4 s + e.
  const size_t srow = (((size_t)n * p.Hv + h) * p.dv + r0 + row) * kDk + 4 * s;
  float S[kVec][4];
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.state_in) x = __ldg(reinterpret_cast<const float4*>(p.state_in + srow + 32 * m));
    S[m][0] = x.x; S[m][1] = x.y; S[m][2] = x.z; S[m][3] = x.w;
  }

  const int nblocks = (end - beg + kChunk - 1) / kChunk;
  if (nblocks > 0) {
    Prefetch pf;
    load_block(pf, p, h, hk, r0, beg, min(kChunk, end - beg), tid);
    store_block(sm, 0, pf, p.scale, tid);
    __syncthreads();
    block_kq(sm, 0, tid);
    __syncthreads();

    for (int blk = 0; blk < nblocks; ++blk) {
      const int b = blk & 1;
      const int t0 = beg + blk * kChunk;
      const int ntok = min(kChunk, end - t0);
      const bool more = blk + 1 < nblocks;
      if (more) load_block(pf, p, h, hk, r0, t0 + kChunk, min(kChunk, end - t0 - kChunk), tid);

      float4 kk[kVec], qq[kVec];
#pragma unroll
      for (int m = 0; m < kVec; ++m) {
        kk[m] = *reinterpret_cast<const float4*>(&sm.k[b][0][32 * m + 4 * s]);
        qq[m] = *reinterpret_cast<const float4*>(&sm.q[b][0][32 * m + 4 * s]);
      }
      for (int t = 0; t < ntok; ++t) {
        // next token's k and q (the block is zero-padded, so t + 1 < kChunk is enough)
        float4 kn[kVec], qn[kVec];
        const int tn = t + 1 < kChunk ? t + 1 : t;
#pragma unroll
        for (int m = 0; m < kVec; ++m) {
          kn[m] = *reinterpret_cast<const float4*>(&sm.k[b][tn][32 * m + 4 * s]);
          qn[m] = *reinterpret_cast<const float4*>(&sm.q[b][tn][32 * m + 4 * s]);
        }
        float u0 = 0.f, u1 = 0.f, w0 = 0.f, w1 = 0.f;   // S.k and S.q~, two chains each
#pragma unroll
        for (int m = 0; m < kVec; ++m) {
          u0 = fmaf(S[m][0], kk[m].x, u0);
          w0 = fmaf(S[m][0], qq[m].x, w0);
          u1 = fmaf(S[m][1], kk[m].y, u1);
          w1 = fmaf(S[m][1], qq[m].y, w1);
          u0 = fmaf(S[m][2], kk[m].z, u0);
          w0 = fmaf(S[m][2], qq[m].z, w0);
          u1 = fmaf(S[m][3], kk[m].w, u1);
          w1 = fmaf(S[m][3], qq[m].w, w1);
        }
        float u = u0 + u1, w = w0 + w1;
        u += __shfl_xor_sync(0xFFFFFFFFu, u, 1);
        w += __shfl_xor_sync(0xFFFFFFFFu, w, 1);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, 2);
        w += __shfl_xor_sync(0xFFFFFFFFu, w, 2);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, 4);
        w += __shfl_xor_sync(0xFFFFFFFFu, w, 4);

        const float4 sc = sm.sc[b][t];                  // alpha, beta, k . q~
        const float vi = sm.v[b][t][row];
        const float c = sc.y * (vi - sc.x * u);
        if (s == 0) sm.o[t][row] = fmaf(sc.x, w, c * sc.z);
#pragma unroll
        for (int m = 0; m < kVec; ++m) {
          S[m][0] = fmaf(sc.x, S[m][0], c * kk[m].x);
          S[m][1] = fmaf(sc.x, S[m][1], c * kk[m].y);
          S[m][2] = fmaf(sc.x, S[m][2], c * kk[m].z);
          S[m][3] = fmaf(sc.x, S[m][3], c * kk[m].w);
          kk[m] = kn[m];
          qq[m] = qn[m];
        }
      }

      if (more) store_block(sm, b ^ 1, pf, p.scale, tid);
      __syncthreads();
      // o of this block: 32 tokens x 32 rows, 16 bytes per thread of the first half
      if (tid < kThreads / 2) {
        const int tt = tid >> 2, c8 = (tid & 3) * 8;
        if (tt < ntok) {
          const float* src = &sm.o[tt][c8];
          uint4 out;
          out.x = pack_bf16(src[0], src[1]);
          out.y = pack_bf16(src[2], src[3]);
          out.z = pack_bf16(src[4], src[5]);
          out.w = pack_bf16(src[6], src[7]);
          *reinterpret_cast<uint4*>(p.o + ((size_t)(t0 + tt) * p.Hv + h) * p.dv + r0 + c8) = out;
        }
      }
      if (more) block_kq(sm, b ^ 1, tid);
      __syncthreads();
    }
  }

  if (p.state_out) {
#pragma unroll
    for (int m = 0; m < kVec; ++m)
      *reinterpret_cast<float4*>(p.state_out + srow + 32 * m) =
          make_float4(S[m][0], S[m][1], S[m][2], S[m][3]);
  }
}

}  // namespace

cudaError_t launch_gdn_scan(const GdnParams& p, cudaStream_t st) {
  const int smem = (int)sizeof(GdnSmem);
  cudaError_t e = cudaFuncSetAttribute(gdn_scan_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.dv / kRows, p.Hv, p.N);
  gdn_scan_kernel<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
