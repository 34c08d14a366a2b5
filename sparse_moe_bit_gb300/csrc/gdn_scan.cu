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
// a pair of rows, 16 fp32 state values of each, for the whole scan: the
// state never leaves registers until the end, and every k and q value a lane
// reads from shared memory serves two rows.  The four dot products are
// summed across the eight lanes by one shuffle butterfly, after which all
// eight hold the same c (addition is commutative, so the butterfly gives
// every lane identical bits).  A CTA of 128 threads holds 32 rows of one
// head; grid (dv/32, Hv, sequences).  Tokens are staged 32 at a time in
// shared memory as fp32 (k and scaled q, the 32 rows' v values, alpha, beta
// and k . q~ per token), double-buffered: the next block's global loads are
// issued into registers before the current block is scanned and stored to
// the other buffer after.  Lane s holds columns 32 m + 4 s + e (m, e < 4),
// so the eight distinct float4 addresses one warp reads per load cover all
// 32 banks.
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kDk = kGdnDk;             // state columns (key width)
constexpr int kRows = kGdnRows;         // state rows per CTA
constexpr int kLanes = 8;               // lanes per pair of rows
constexpr int kThreads = kRows / 2 * kLanes;  // 128
constexpr int kChunk = 32;              // tokens per staged block
constexpr int kVec = kDk / (4 * kLanes);  // float4 groups per lane (4)
constexpr int kKQ = kChunk * kDk / 8 / kThreads;  // 16-byte pieces of k (and q) per thread

static_assert(kThreads == 128 && kVec == 4 && kKQ == 4, "layout below assumes these");
static_assert(kChunk * kRows / 8 == kThreads, "one 16-byte piece of v (and of o) per thread");

struct __align__(16) GdnSmem {
  float k[2][kChunk][kDk];
  float q[2][kChunk][kDk];       // scaled by the readout scale
  float v[2][kChunk][kRows];
  float4 sc[2][kChunk];          // alpha, beta, k . q~, unused
  float o[kChunk][kRows];
};

// One staged block, in flight in registers.
struct Prefetch {
  uint4 k[kKQ], q[kKQ], v;
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

// Issue the global loads of tokens t0 .. t0+n-1 (n <= kChunk; pieces past n
// load nothing and hold zeros).
__device__ __forceinline__ void load_block(Prefetch& pf, const GdnParams& p, int h, int hk,
                                           int r0, int t0, int n, int tid) {
#pragma unroll
  for (int j = 0; j < kKQ; ++j) {
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
  {
    const int tt = tid >> 2, c8 = (tid & 3) * 8;
    pf.v = make_uint4(0, 0, 0, 0);
    if (tt < n)
      pf.v = __ldg(reinterpret_cast<const uint4*>(p.v + ((size_t)(t0 + tt) * p.Hv + h) * p.dv +
                                                  r0 + c8));
  }
  pf.gb = 0.f;
  if (tid < 2 * kChunk) {
    const int tt = tid & (kChunk - 1);
    if (tt < n) {
      const size_t off = (size_t)(t0 + tt) * p.Hv + h;
      pf.gb = tid >= kChunk ? __ldg(p.beta + off) : __ldg(p.g + off);
    }
  }
}

__device__ __forceinline__ void store_block(GdnSmem& sm, int b, const Prefetch& pf, float scale,
                                            int tid) {
#pragma unroll
  for (int j = 0; j < kKQ; ++j) {
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
  {
    const int tt = tid >> 2, c8 = (tid & 3) * 8;
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(&pf.v);
    float4* vd = reinterpret_cast<float4*>(&sm.v[b][tt][c8]);
    vd[0] = make_float4(bf16_lo(vw[0]), bf16_hi(vw[0]), bf16_lo(vw[1]), bf16_hi(vw[1]));
    vd[1] = make_float4(bf16_lo(vw[2]), bf16_hi(vw[2]), bf16_lo(vw[3]), bf16_hi(vw[3]));
  }
  if (tid < kChunk)
    sm.sc[b][tid].x = expf(pf.gb);                       // alpha, fp32
  else if (tid < 2 * kChunk)
    sm.sc[b][tid - kChunk].y = pf.gb;                    // beta
}

// k . q~ of each staged token: eight threads per token (two tokens per
// thread), same column split as the state rows.
__device__ __forceinline__ void block_kq(GdnSmem& sm, int b, int tid) {
  const int s = tid & 7;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int tt = (tid >> 3) + half * (kChunk / 2);
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
}

__device__ __forceinline__ void load_kq(const GdnSmem& sm, int b, int t, int s, float4 (&kk)[kVec],
                                        float4 (&qq)[kVec]) {
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    kk[m] = *reinterpret_cast<const float4*>(&sm.k[b][t][32 * m + 4 * s]);
    qq[m] = *reinterpret_cast<const float4*>(&sm.q[b][t][32 * m + 4 * s]);
  }
}

// One token for the lane's two rows (2 pr, 2 pr + 1).
__device__ __forceinline__ void scan_token(GdnSmem& sm, int b, int t, int pr, int s,
                                           float (&SA)[kVec][4], float (&SB)[kVec][4],
                                           const float4 (&kk)[kVec], const float4 (&qq)[kVec]) {
  float uA0 = 0.f, uA1 = 0.f, wA0 = 0.f, wA1 = 0.f;   // S.k and S.q~ of row A, two chains each
  float uB0 = 0.f, uB1 = 0.f, wB0 = 0.f, wB1 = 0.f;
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    uA0 = fmaf(SA[m][0], kk[m].x, uA0);
    wA0 = fmaf(SA[m][0], qq[m].x, wA0);
    uB0 = fmaf(SB[m][0], kk[m].x, uB0);
    wB0 = fmaf(SB[m][0], qq[m].x, wB0);
    uA1 = fmaf(SA[m][1], kk[m].y, uA1);
    wA1 = fmaf(SA[m][1], qq[m].y, wA1);
    uB1 = fmaf(SB[m][1], kk[m].y, uB1);
    wB1 = fmaf(SB[m][1], qq[m].y, wB1);
    uA0 = fmaf(SA[m][2], kk[m].z, uA0);
    wA0 = fmaf(SA[m][2], qq[m].z, wA0);
    uB0 = fmaf(SB[m][2], kk[m].z, uB0);
    wB0 = fmaf(SB[m][2], qq[m].z, wB0);
    uA1 = fmaf(SA[m][3], kk[m].w, uA1);
    wA1 = fmaf(SA[m][3], qq[m].w, wA1);
    uB1 = fmaf(SB[m][3], kk[m].w, uB1);
    wB1 = fmaf(SB[m][3], qq[m].w, wB1);
  }
  float uA = uA0 + uA1, wA = wA0 + wA1, uB = uB0 + uB1, wB = wB0 + wB1;
#pragma unroll
  for (int lv = 1; lv < kLanes; lv <<= 1) {
    uA += __shfl_xor_sync(0xFFFFFFFFu, uA, lv);
    wA += __shfl_xor_sync(0xFFFFFFFFu, wA, lv);
    uB += __shfl_xor_sync(0xFFFFFFFFu, uB, lv);
    wB += __shfl_xor_sync(0xFFFFFFFFu, wB, lv);
  }
  const float4 sc = sm.sc[b][t];                        // alpha, beta, k . q~
  const float2 vv = *reinterpret_cast<const float2*>(&sm.v[b][t][2 * pr]);
  const float cA = sc.y * (vv.x - sc.x * uA);
  const float cB = sc.y * (vv.y - sc.x * uB);
  if (s == 0)
    *reinterpret_cast<float2*>(&sm.o[t][2 * pr]) =
        make_float2(fmaf(sc.x, wA, cA * sc.z), fmaf(sc.x, wB, cB * sc.z));
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    SA[m][0] = fmaf(sc.x, SA[m][0], cA * kk[m].x);
    SA[m][1] = fmaf(sc.x, SA[m][1], cA * kk[m].y);
    SA[m][2] = fmaf(sc.x, SA[m][2], cA * kk[m].z);
    SA[m][3] = fmaf(sc.x, SA[m][3], cA * kk[m].w);
    SB[m][0] = fmaf(sc.x, SB[m][0], cB * kk[m].x);
    SB[m][1] = fmaf(sc.x, SB[m][1], cB * kk[m].y);
    SB[m][2] = fmaf(sc.x, SB[m][2], cB * kk[m].z);
    SB[m][3] = fmaf(sc.x, SB[m][3], cB * kk[m].w);
  }
}

__global__ void __launch_bounds__(kThreads, 1) gdn_scan_kernel(const GdnParams p) {
  extern __shared__ float4 gdn_smem_raw[];
  GdnSmem& sm = *reinterpret_cast<GdnSmem*>(gdn_smem_raw);
  const int tid = threadIdx.x;
  const int pr = tid >> 3, s = tid & 7;                 // row pair, lane within it
  const int r0 = blockIdx.x * kRows, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);

  int beg = 0, end = p.T;
  if (p.offsets) {
    beg = min(max(__ldg(p.offsets + n), 0), p.T);
    end = min(max(__ldg(p.offsets + n + 1), beg), p.T);
  }

  // 16 state values of each of the two rows: columns 32 m + 4 s + e.
  const size_t srow = (((size_t)n * p.Hv + h) * p.dv + r0 + 2 * pr) * kDk + 4 * s;
  float SA[kVec][4], SB[kVec][4];
#pragma unroll
  for (int m = 0; m < kVec; ++m) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
    if (p.state_in) {
      a = __ldg(reinterpret_cast<const float4*>(p.state_in + srow + 32 * m));
      c = __ldg(reinterpret_cast<const float4*>(p.state_in + srow + kDk + 32 * m));
    }
    SA[m][0] = a.x; SA[m][1] = a.y; SA[m][2] = a.z; SA[m][3] = a.w;
    SB[m][0] = c.x; SB[m][1] = c.y; SB[m][2] = c.z; SB[m][3] = c.w;
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

      // Two tokens per iteration, k and q of the next token loaded during
      // the current one (the block is zero-padded up to kChunk tokens).
      float4 k0[kVec], q0[kVec], k1[kVec], q1[kVec];
      load_kq(sm, b, 0, s, k0, q0);
      int t = 0;
      for (; t + 1 < ntok; t += 2) {
        load_kq(sm, b, t + 1, s, k1, q1);
        scan_token(sm, b, t, pr, s, SA, SB, k0, q0);
        if (t + 2 < kChunk) load_kq(sm, b, t + 2, s, k0, q0);
        scan_token(sm, b, t + 1, pr, s, SA, SB, k1, q1);
      }
      if (t < ntok) scan_token(sm, b, t, pr, s, SA, SB, k0, q0);

      if (more) store_block(sm, b ^ 1, pf, p.scale, tid);
      __syncthreads();
      // o of this block: 32 tokens x 32 rows, one 16-byte piece per thread
      {
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
    for (int m = 0; m < kVec; ++m) {
      *reinterpret_cast<float4*>(p.state_out + srow + 32 * m) =
          make_float4(SA[m][0], SA[m][1], SA[m][2], SA[m][3]);
      *reinterpret_cast<float4*>(p.state_out + srow + kDk + 32 * m) =
          make_float4(SB[m][0], SB[m][1], SB[m][2], SB[m][3]);
    }
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
