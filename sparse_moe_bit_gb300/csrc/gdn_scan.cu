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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

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


// ---------------------------------------------------------------------------
// Chunked evaluation on the tensor cores (the blockwise way the pages
// mention).  Unrolling the rule over a chunk of C tokens that starts from
// state S_0, with gamma_i the product of the gates up to token i (within the
// chunk) and c_i = beta_i (v_i - alpha_i S_{i-1} k_i):
//     S_i = gamma_i S_0 + sum_{j<=i} (gamma_i / gamma_j) c_j k_j^T,
// so the c vectors solve the unit lower-triangular system (I + L) C = R,
//     L_ij = beta_i (gamma_i / gamma_j) k_i . k_j  (j < i),
//     R_i  = beta_i (v_i - gamma_i S_0 k_i),
// and o_i = scale (gamma_i S_0 q_i + sum_{j<=i} (gamma_i / gamma_j)(q_i . k_j) c_j),
//     S_C = gamma_C S_0 + sum_j (gamma_C / gamma_j) c_j k_j^T.
// Per chunk and CTA (32 state rows of one head): K K^T and Q K^T, (I + L)^-1
// by forward substitution (one lane per column), K S^T and Q S^T, C =
// (I + L)^-1 R, M C with M_ij = (gamma_i / gamma_j) q_i . k_j (j <= i), and
// the state update, all products but the inverse on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation).  q and k are bf16
// already; every fp32 operand enters as a sum of bf16 parts (the state as
// three, the others as two, their products' largest cross terms kept), so
// that the products keep fp32-level accuracy.  The state stays in registers
// for the whole scan as the accumulator fragments of the update's product.
// Gates enter as exp of differences of the chunk's cumulative log gates
// (ratios <= 1: no overflow).  Chunk boundaries follow the call's tokens.
constexpr int kC = 32;      // tokens per chunk (= kChunk, the staging block)
constexpr int kLdA = 136;   // bf16 row pitch of [32][128] operands (68 words apart)
constexpr int kLd32 = 40;   // bf16 row pitch of [*][32] operands (20 words apart)
constexpr int kLdF = 33;    // fp32 row pitch of [32][32] matrices
constexpr int kLdL = 36;    // fp32 row pitch of L (16-byte rows: read a row at a time)
static_assert(kC == kChunk, "the staging block is one chunk");

// One chunk's inputs and input-only matrices (written by the preparing
// warps, read by the state pass one chunk later).
struct __align__(16) ChunkIn {
  uint16_t K[kC][kLdA];                    // k rows [t][c]
  uint16_t Q[kC][kLdA];                    // q rows [t][c] (unscaled)
  uint16_t Kt[kDk][kLd32];                 // k transposed [c][t]
  uint16_t Th[kC][kLd32], Tl[kC][kLd32];   // (I + L)^-1 parts [i][j]
  uint16_t Mh[kC][kLd32], Ml[kC][kLd32];   // M parts [i][j]
  float V[kC][kLdF];                       // v [t][r]
  float beta[kC], eg[kC], fac[kC];         // beta_t, gamma_t, gamma_C / gamma_t
};
struct __align__(16) ChunkSmem {
  ChunkIn in[2];
  // preparing warps' scratch
  float L[kC][kLdL];                       // K K^T, then L
  float QK[kC][kLdF];                      // Q K^T
  float cs[kC];                            // cumulative log gate (0 past the chunk)
  // state pass
  uint16_t S3[3][kRows][kLdA];             // the state slice as bf16 parts hi, mid, lo [r][c]
  uint16_t Rh[kRows][kLd32], Rl[kRows][kLd32];  // R transposed [r][j]
  uint16_t Ch[kRows][kLd32], Cl[kRows][kLd32];  // C transposed [r][j]
  uint16_t Fh[kRows][kLd32], Fl[kRows][kLd32];  // (gamma_C / gamma_j) C transposed [r][j]
  float KS[kC][kLdF], QS[kC][kLdF];        // K S^T, Q S^T [t][r] (QS then o)
};
constexpr int kCThreads = 2 * kThreads;   // warps 0-3: the state pass; 4-7: the next chunk

// barrier of one group of four warps (id 1: state pass, 2: preparing warps)
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kThreads) : "memory");
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
// x = hi + lo (+ the rounding of lo)
__device__ __forceinline__ void split2(float x, uint16_t& h, uint16_t& l) {
  h = bf16_bits(x);
  l = bf16_bits(x - bf16_val(h));
}

// d += a * b for a 16x16 (row-major) and a 16x8 (col-major) bf16 tile
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A fragment of the 16x16 tile at (r0, k0) of a row-major bf16 matrix
__device__ __forceinline__ void frag_a(const uint16_t* A, int ld, int r0, int k0, int lane,
                                       uint32_t (&a)[4]) {
  const uint16_t* p = A + (r0 + (lane >> 2)) * ld + k0 + 2 * (lane & 3);
  a[0] = *reinterpret_cast<const uint32_t*>(p);
  a[1] = *reinterpret_cast<const uint32_t*>(p + 8 * ld);
  a[2] = *reinterpret_cast<const uint32_t*>(p + 8);
  a[3] = *reinterpret_cast<const uint32_t*>(p + 8 * ld + 8);
}
// B fragment of the 16x8 tile at (k0, n0) of a matrix stored as [n][k]
__device__ __forceinline__ void frag_b(const uint16_t* B, int ld, int k0, int n0, int lane,
                                       uint32_t (&b)[2]) {
  const uint16_t* p = B + (n0 + (lane >> 2)) * ld + k0 + 2 * (lane & 3);
  b[0] = *reinterpret_cast<const uint32_t*>(p);
  b[1] = *reinterpret_cast<const uint32_t*>(p + 8);
}
// a 16x8 fp32 accumulator tile at (r0, n0) of a matrix of row pitch ld
__device__ __forceinline__ void store_acc(float* D, int ld, int r0, int n0, int lane,
                                          const float (&d)[4]) {
  const int g = lane >> 2, t2 = 2 * (lane & 3);
  D[(r0 + g) * ld + n0 + t2] = d[0];
  D[(r0 + g) * ld + n0 + t2 + 1] = d[1];
  D[(r0 + g + 8) * ld + n0 + t2] = d[2];
  D[(r0 + g + 8) * ld + n0 + t2 + 1] = d[3];
}

// Warps 4-7 (thread pt = 0..127): one chunk's inputs into B (the staged
// loads in pf), its gates, K K^T and Q K^T, L and M, and (I + L)^-1.
__device__ __forceinline__ void prep_chunk(ChunkSmem& sm, ChunkIn& B, const Prefetch& pf,
                                           int pt) {
  const int pw = pt >> 5, lane = pt & 31;
  // ---- stage: k and q rows, v, the gates (a warp scan of the log gates), beta
#pragma unroll
  for (int j = 0; j < kKQ; ++j) {
    const int i = pt + j * kThreads;
    const int tt = i >> 4, c8 = (i & 15) * 8;
    *reinterpret_cast<uint4*>(&B.K[tt][c8]) = pf.k[j];
    *reinterpret_cast<uint4*>(&B.Q[tt][c8]) = pf.q[j];
  }
  {
    const int tt = pt >> 2, c8 = (pt & 3) * 8;
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(&pf.v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      B.V[tt][c8 + 2 * e] = bf16_lo(vw[e]);
      B.V[tt][c8 + 2 * e + 1] = bf16_hi(vw[e]);
    }
  }
  if (pw == 0) {  // thread t holds g of token t
    float c = pf.gb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xFFFFFFFFu, c, o);
      if (lane >= o) c += u;
    }
    const float cl = __shfl_sync(0xFFFFFFFFu, c, kC - 1);
    sm.cs[lane] = c;
    B.eg[lane] = expf(c);
    B.fac[lane] = expf(cl - c);
  } else if (pw == 1) {  // thread 32 + t holds beta of token t
    B.beta[lane] = pf.gb;
  }
  group_sync(2);
  // ---- k transposed (thread = column c), K K^T (warps 0, 1) and Q K^T (2, 3)
#pragma unroll
  for (int tp = 0; tp < kC / 2; ++tp)
    *reinterpret_cast<uint32_t*>(&B.Kt[pt][2 * tp]) =
        (uint32_t)B.K[2 * tp][pt] | ((uint32_t)B.K[2 * tp + 1][pt] << 16);
  {
    const uint16_t* A = (pw < 2) ? &B.K[0][0] : &B.Q[0][0];
    float* D = (pw < 2) ? &sm.L[0][0] : &sm.QK[0][0];
    const int ld = (pw < 2) ? kLdL : kLdF;
    const int m0 = 16 * (pw & 1);
    float d[4][4] = {};
#pragma unroll
    for (int k0 = 0; k0 < kDk; k0 += 16) {
      uint32_t a[4];
      frag_a(A, kLdA, m0, k0, lane, a);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t b[2];
        frag_b(&B.K[0][0], kLdA, k0, 8 * nt, lane, b);
        mma_bf16(d[nt], a, b);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) store_acc(D, ld, m0, 8 * nt, lane, d[nt]);
  }
  group_sync(2);
  // ---- L (in place) and M's parts: element (i, j) = (pw + 4 m, lane); loads first
  {
    const int j = lane;
    const float csj = sm.cs[j];
    float kk[8], qk[8], bi[8], csi[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int i = pw + 4 * m;
      kk[m] = sm.L[i][j];
      qk[m] = sm.QK[i][j];
      bi[m] = B.beta[i];
      csi[m] = sm.cs[i];
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int i = pw + 4 * m;
      // gamma_i / gamma_j = exp(cs_i - cs_j) <= 1 where it is used (j <= i)
      const float rij = expf(fminf(csi[m] - csj, 0.f));
      const float l = (j < i) ? bi[m] * rij * kk[m] : 0.f;
      const float mm = (j <= i) ? rij * qk[m] : 0.f;
      sm.L[i][j] = l;
      uint16_t mh, ml;
      split2(mm, mh, ml);
      B.Mh[i][j] = mh;
      B.Ml[i][j] = ml;
    }
  }
  group_sync(2);
  // ---- (I + L)^-1 by forward substitution, lane = column (warp 4)
  if (pw == 0) {
    float x[kC];
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      // row i of L, a 16-byte piece at a time (every lane reads the same row)
      float li[kC];
#pragma unroll
      for (int j4 = 0; j4 < (i + 3) / 4; ++j4) {
        const float4 q4 = *reinterpret_cast<const float4*>(&sm.L[i][4 * j4]);
        li[4 * j4] = q4.x;
        li[4 * j4 + 1] = q4.y;
        li[4 * j4 + 2] = q4.z;
        li[4 * j4 + 3] = q4.w;
      }
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) {
        if ((j & 3) == 0) s0 = fmaf(li[j], x[j], s0);
        else if ((j & 3) == 1) s1 = fmaf(li[j], x[j], s1);
        else if ((j & 3) == 2) s2 = fmaf(li[j], x[j], s2);
        else s3 = fmaf(li[j], x[j], s3);
      }
      x[i] = ((i == lane) ? 1.f : 0.f) - ((s0 + s1) + (s2 + s3));
    }
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      uint16_t th, tl;
      split2(x[i], th, tl);
      B.Th[i][lane] = th;
      B.Tl[i][lane] = tl;
    }
  }
}

__global__ void __launch_bounds__(kCThreads, 1) gdn_chunk_kernel(const GdnParams p) {
  extern __shared__ float4 gdn_smem_raw[];
  ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(gdn_smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool prep = warp >= 4;
  const int g4 = lane >> 2, t2 = 2 * (lane & 3);
  const int r0 = blockIdx.x * kRows, h = blockIdx.y, n = blockIdx.z;
  const int hk = h / (p.Hv / p.Hk);

  int beg = 0, end = p.T;
  if (p.offsets) {
    beg = min(max(__ldg(p.offsets + n), 0), p.T);
    end = min(max(__ldg(p.offsets + n + 1), beg), p.T);
  }
  const int nblocks = (end - beg + kC - 1) / kC;
  auto ntok_of = [&](int blk) { return min(kC, end - beg - blk * kC); };

  // The state slice S[r][c] (r < 32 of this CTA), in warps 0-3, as the
  // accumulators of the update's product: warp w holds columns 32 w .. 32 w
  // + 31 of both 16-row halves, tile (mt, nt) element e at row 16 mt + g4
  // (+8 for e >= 2), column 32 w + 8 nt + t2 (+1 for odd e).
  float Sacc[2][4][4];
  const size_t sbase = (((size_t)n * p.Hv + h) * p.dv + r0) * kDk;
  if (!prep) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 16 * mt + g4 + 8 * (e >> 1), c = 32 * warp + 8 * nt + t2 + (e & 1);
          Sacc[mt][nt][e] = p.state_in ? __ldg(p.state_in + sbase + (size_t)r * kDk + c) : 0.f;
        }
  }

  Prefetch pf;
  if (prep && nblocks > 0) {
    const int pt = tid - kThreads;
    load_block(pf, p, h, hk, r0, beg, ntok_of(0), pt);
    prep_chunk(sm, sm.in[0], pf, pt);
    if (nblocks > 1) load_block(pf, p, h, hk, r0, beg + kC, ntok_of(1), pt);
  }
  __syncthreads();

  for (int blk = 0; blk < nblocks; ++blk) {
    if (prep) {
      // the next chunk's inputs and matrices, and the loads of the one after
      if (blk + 1 < nblocks) {
        const int pt = tid - kThreads;
        prep_chunk(sm, sm.in[(blk + 1) & 1], pf, pt);
        if (blk + 2 < nblocks)
          load_block(pf, p, h, hk, r0, beg + (blk + 2) * kC, ntok_of(blk + 2), pt);
      }
    } else {
      const ChunkIn& B = sm.in[blk & 1];
      const int t0 = beg + blk * kC, ntok = ntok_of(blk);
      // ---- the state's bf16 parts
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 16 * mt + g4 + 8 * (e >> 1), c = 32 * warp + 8 * nt + t2 + (e & 1);
            const float x = Sacc[mt][nt][e];
            const uint16_t hi = bf16_bits(x);
            const float r1 = x - bf16_val(hi);
            const uint16_t mid = bf16_bits(r1);
            sm.S3[0][r][c] = hi;
            sm.S3[1][r][c] = mid;
            sm.S3[2][r][c] = bf16_bits(r1 - bf16_val(mid));
          }
      group_sync(1);
      // ---- K S^T (warps 0, 1) and Q S^T (2, 3): rows 16 (w & 1), 4 column tiles
      {
        const uint16_t* A = (warp < 2) ? &B.K[0][0] : &B.Q[0][0];
        float* D = (warp < 2) ? &sm.KS[0][0] : &sm.QS[0][0];
        const int m0 = 16 * (warp & 1);
        float d[4][4] = {};
#pragma unroll
        for (int k0 = 0; k0 < kDk; k0 += 16) {
          uint32_t a[4];
          frag_a(A, kLdA, m0, k0, lane, a);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              uint32_t b[2];
              frag_b(&sm.S3[part][0][0], kLdA, k0, 8 * nt, lane, b);
              mma_bf16(d[nt], a, b);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) store_acc(D, kLdF, m0, 8 * nt, lane, d[nt]);
      }
      group_sync(1);
      // ---- R = beta (V - gamma K S^T), transposed parts [r][j]; loads first
      {
        float rr[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int jt = warp + 4 * m, r = lane;
          rr[m] = B.beta[jt] * (B.V[jt][r] - B.eg[jt] * sm.KS[jt][r]);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int jt = warp + 4 * m, r = lane;
          uint16_t rh, rl;
          split2(rr[m], rh, rl);
          sm.Rh[r][jt] = rh;
          sm.Rl[r][jt] = rl;
        }
      }
      group_sync(1);
      // ---- C = (I + L)^-1 R: warp w rows 16 (w >> 1), columns 16 (w & 1) ..
      {
        const int m0 = 16 * (warp >> 1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int n0 = 16 * (warp & 1) + 8 * nt;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          float d2[4] = {0.f, 0.f, 0.f, 0.f};  // the small cross terms, a second chain
#pragma unroll
          for (int k0 = 0; k0 < kC; k0 += 16) {
            uint32_t ah[4], al[4], bh[2], bl[2];
            frag_a(&B.Th[0][0], kLd32, m0, k0, lane, ah);
            frag_a(&B.Tl[0][0], kLd32, m0, k0, lane, al);
            frag_b(&sm.Rh[0][0], kLd32, k0, n0, lane, bh);
            frag_b(&sm.Rl[0][0], kLd32, k0, n0, lane, bl);
            mma_bf16(d2, al, bh);
            mma_bf16(d2, ah, bl);
            mma_bf16(d, ah, bh);
          }
          // C's parts [r][j], and (gamma_C / gamma_j) C's parts
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jt = m0 + g4 + 8 * (e >> 1), r = n0 + t2 + (e & 1);
            const float cv = d[e] + d2[e];
            uint16_t ch, cl, fh, fl;
            split2(cv, ch, cl);
            split2(B.fac[jt] * cv, fh, fl);
            sm.Ch[r][jt] = ch;
            sm.Cl[r][jt] = cl;
            sm.Fh[r][jt] = fh;
            sm.Fl[r][jt] = fl;
          }
        }
      }
      group_sync(1);
      // ---- o = scale (gamma Q S^T + M C), staged in QS
      {
        const int m0 = 16 * (warp >> 1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int n0 = 16 * (warp & 1) + 8 * nt;
          float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k0 = 0; k0 < kC; k0 += 16) {
            uint32_t ah[4], al[4], bh[2], bl[2];
            frag_a(&B.Mh[0][0], kLd32, m0, k0, lane, ah);
            frag_a(&B.Ml[0][0], kLd32, m0, k0, lane, al);
            frag_b(&sm.Ch[0][0], kLd32, k0, n0, lane, bh);
            frag_b(&sm.Cl[0][0], kLd32, k0, n0, lane, bl);
            mma_bf16(d2, al, bh);
            mma_bf16(d2, ah, bl);
            mma_bf16(d, ah, bh);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = m0 + g4 + 8 * (e >> 1), r = n0 + t2 + (e & 1);
            sm.QS[t][r] = p.scale * fmaf(B.eg[t], sm.QS[t][r], d[e] + d2[e]);
          }
        }
      }
      // ---- state: S <- gamma_C S + (gamma_C / gamma_j) C^T K (two parts of
      //      the left factor, k exact)
      {
        const float gC = B.eg[kC - 1];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) Sacc[mt][nt][e] *= gC;
#pragma unroll
        for (int k0 = 0; k0 < kC; k0 += 16) {
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            uint32_t ah[4], al[4];
            frag_a(&sm.Fh[0][0], kLd32, 16 * mt, k0, lane, ah);
            frag_a(&sm.Fl[0][0], kLd32, 16 * mt, k0, lane, al);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              uint32_t b[2];
              frag_b(&B.Kt[0][0], kLd32, k0, 32 * warp + 8 * nt, lane, b);
              mma_bf16(Sacc[mt][nt], al, b);
              mma_bf16(Sacc[mt][nt], ah, b);
            }
          }
        }
      }
      group_sync(1);
      // ---- o of the chunk's tokens: one 16-byte piece (8 rows) per thread
      {
        const int tt = tid >> 2, c8 = (tid & 3) * 8;
        if (tt < ntok) {
          const float* src = &sm.QS[tt][c8];
          uint4 out;
          out.x = pack_bf16(src[0], src[1]);
          out.y = pack_bf16(src[2], src[3]);
          out.z = pack_bf16(src[4], src[5]);
          out.w = pack_bf16(src[6], src[7]);
          *reinterpret_cast<uint4*>(p.o + ((size_t)(t0 + tt) * p.Hv + h) * p.dv + r0 + c8) = out;
        }
      }
    }
    __syncthreads();  // chunk blk done, chunk blk + 1 prepared
  }

  if (!prep && p.state_out) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 16 * mt + g4 + 8 * (e >> 1), c = 32 * warp + 8 * nt + t2 + (e & 1);
          p.state_out[sbase + (size_t)r * kDk + c] = Sacc[mt][nt][e];
        }
  }
}

}  // namespace

cudaError_t launch_gdn_scan(const GdnParams& p, cudaStream_t st) {
  const dim3 grid(p.dv / kRows, p.Hv, p.N);
  static const bool token_loop = getenv("MOE_GDN_TOKEN_LOOP") != nullptr;
  if (token_loop) {
    const int smem = (int)sizeof(GdnSmem);
    cudaError_t e = cudaFuncSetAttribute(gdn_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(gdn_scan_kernel, grid, dim3(kThreads), smem, st, p);
  }
  {
    const int smem = (int)sizeof(ChunkSmem);
    cudaError_t e = cudaFuncSetAttribute(gdn_chunk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(gdn_chunk_kernel, grid, dim3(kCThreads), smem, st, p);
  }
}

}  // namespace moe
