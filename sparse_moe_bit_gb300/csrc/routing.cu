// GPU-resident routing: softmax/top-k, histogram, prefix scan, scatter and
// tile (block) map, and the deterministic combine.  No host round-trip: every
// size the later kernels need stays in device memory.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Keep expert routing on the GPU" (histogram of assignments per expert,
// prefix scan to start offsets, scatter of rows into their expert groups,
// block map of the fixed-size blocks the grouped GEMM processes) and
// §"Match tile size to expert load" (tiles sized from the expert's rows).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>
#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"
#include "softmax_df.cuh"
#include "topk_warp.cuh"

namespace moe {
namespace {

// Top-k selection (topk_warp): the router's K-split partial logits are
// summed in a fixed order, the bias added, and the top k kept by (logit
// desc, index asc); lane l holds the order keys of experts l, l+32, ...; each
// round every lane finds its best key not yet taken (first slot among equal
// keys, i.e. the lowest index), the warp maximum of those and then the
// smallest expert index among the lanes holding it name the winner (two warp
// reductions per round).
constexpr int kTopkThreads = 32 * kTokPerBlock;
static_assert(kTopkThreads <= 1024, "one warp per token of a block");

// Top-k of token t by one warp (t < T checked by the caller): the fixed-order
// sum of the K-split partial logits and the bias, the logits row, the kept
// experts idx[t][0..k) in order, their logits into s_vw[0..k) and one count
// per kept expert into the block histogram cnt.
template <int VPL>
__device__ __forceinline__ void topk_warp(const float* __restrict__ part, int KS, int T, int E,
                                          int k, const float* __restrict__ bias,
                                          float* __restrict__ logits, int32_t* __restrict__ idx_out,
                                          int t, float* s_vw, int* cnt, int* err) {
  const int lane = threadIdx.x & 31;
  float v[VPL];
  uint32_t key[VPL];
  bool nan_seen = false;
  // all of the lane's loads first (one round trip for up to kKsBatch
  // splits), then the sums in the fixed order 0 + part_0 + part_1 + ... + bias
  constexpr int kKsBatch = VPL <= 8 ? 4 : 2;
  float pa[VPL], ba[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    ba[j] = (e < E && bias) ? __ldg(bias + e) : 0.0f;
    pa[j] = 0.0f;
  }
  for (int q0 = 0; q0 < KS; q0 += kKsBatch) {
    float pq[kKsBatch][VPL];
#pragma unroll
    for (int qq = 0; qq < kKsBatch; ++qq)
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        pq[qq][j] = (e < E && q0 + qq < KS)
                        ? __ldg(part + ((long long)(q0 + qq) * T + t) * E + e) : 0.0f;
      }
#pragma unroll
    for (int qq = 0; qq < kKsBatch; ++qq)
      if (q0 + qq < KS)
#pragma unroll
        for (int j = 0; j < VPL; ++j) pa[j] += pq[qq][j];
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    float s = -INFINITY;
    uint32_t kk = 0u;  // empty; every real key is larger
    if (e < E) {
      s = 0.0f + pa[j];
      if (bias) s += ba[j];
      logits[(long long)t * E + e] = s;
      if (s != s) {
        nan_seen = true;
        s = -INFINITY;
      }
      kk = ord_key(s);
    }
    v[j] = s;
    key[j] = kk;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(err, MOE_DEVERR_NAN_LOGIT);

  // lane r keeps the r-th choice
  float my_v = -INFINITY;
  int my_e = 0;
  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0u;
    int bj = 0;
    float bv = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const bool better = key[j] > bk;
      bk = better ? key[j] : bk;
      bv = better ? v[j] : bv;
      bj = better ? j : bj;
    }
    const uint32_t M = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t win =
        __reduce_min_sync(0xffffffffu, bk == M ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
    const float wv = __shfl_sync(0xffffffffu, bv, (int)(win & 31u));
    if ((int)(win & 31u) == lane) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) key[j] = (j == (int)(win >> 5)) ? 0u : key[j];
    }
    if (lane == r) {
      my_v = wv;
      my_e = (int)win;
    }
  }
  if (lane < k) {
    idx_out[(long long)t * k + lane] = my_e;
    s_vw[lane] = my_v;
    atomicAdd(&cnt[my_e], 1);
  }
}

// topk_warp for E <= 256 with lane l holding experts 8l .. 8l+7 (contiguous
// loads; the ranking of warp_topk_lists): the same fixed-order sums, outputs
// and counts.
__device__ __forceinline__ void topk_warp8(const float* __restrict__ part, int KS, int T, int E,
                                           int k, const float* __restrict__ bias,
                                           float* __restrict__ logits,
                                           int32_t* __restrict__ idx_out, int t, float* s_vw,
                                           int* cnt, int* err) {
  const int lane = threadIdx.x & 31;
  const int e0 = 8 * lane;
  const bool vec = (E & 7) == 0;  // whole 32-byte groups: vector loads
  float pa[8], ba[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    pa[i] = 0.0f;
    ba[i] = 0.0f;
  }
  if (bias && e0 < E) {
    if (vec) {
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(bias + e0));
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(bias + e0) + 1);
      ba[0] = b0.x; ba[1] = b0.y; ba[2] = b0.z; ba[3] = b0.w;
      ba[4] = b1.x; ba[5] = b1.y; ba[6] = b1.z; ba[7] = b1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) ba[i] = (e0 + i < E) ? __ldg(bias + e0 + i) : 0.0f;
    }
  }
  // the lane's loads of two splits at a time, then the sums in the fixed
  // order 0 + part_0 + part_1 + ... + bias
  for (int q0 = 0; q0 < KS; q0 += 2) {
    float pq[2][8];
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const float* src = part + ((long long)(q0 + qq) * T + t) * E + e0;
      const bool on = q0 + qq < KS && e0 < E;
      if (vec) {
        const float4 a0 = on ? __ldg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 a1 = on ? __ldg(reinterpret_cast<const float4*>(src) + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        pq[qq][0] = a0.x; pq[qq][1] = a0.y; pq[qq][2] = a0.z; pq[qq][3] = a0.w;
        pq[qq][4] = a1.x; pq[qq][5] = a1.y; pq[qq][6] = a1.z; pq[qq][7] = a1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) pq[qq][i] = (on && e0 + i < E) ? __ldg(src + i) : 0.0f;
      }
    }
#pragma unroll
    for (int qq = 0; qq < 2; ++qq)
      if (q0 + qq < KS)
#pragma unroll
        for (int i = 0; i < 8; ++i) pa[i] += pq[qq][i];
  }
  bool nan_seen = false;
  unsigned long long s8[8];
  float lv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e0 + i;
    float s = 0.0f + pa[i];
    if (bias) s += ba[i];
    lv[i] = s;
    if (s != s) {
      nan_seen = true;
      s = -INFINITY;
    }
    s8[i] = (e < E) ? (((unsigned long long)ord_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)e))
                    : 0ull;
  }
  float* lo = logits + (long long)t * E + e0;
  if (vec) {
    if (e0 < E) {
      reinterpret_cast<float4*>(lo)[0] = make_float4(lv[0], lv[1], lv[2], lv[3]);
      reinterpret_cast<float4*>(lo)[1] = make_float4(lv[4], lv[5], lv[6], lv[7]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (e0 + i < E) lo[i] = lv[i];
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(err, MOE_DEVERR_NAN_LOGIT);
  const unsigned long long kw = warp_topk_lists(s8, k, lane);
  if (lane < k) {
    const int my_e = (int)(0xFFFFFFFFu - (uint32_t)kw);
    idx_out[(long long)t * k + lane] = my_e;
    s_vw[lane] = ord_value((uint32_t)(kw >> 32));
    atomicAdd(&cnt[my_e], 1);
  }
}

// Routing weights of the tokens tb .. tb + kTokPerBlock - 1 (those < tend)
// from their kept logits s_v (after a __syncthreads): w_r = exp(l_r - l_0) /
// sum_i exp(l_i - l_0) in double-float arithmetic (within one ulp of the fp64
// value; see softmax_df.cuh); with infinite logits the limit: +inf experts
// share equally, all -inf share equally.  A warp takes 32 / kp tokens at once
// (lane: token, slot), kp = 8 or 16 >= k; the sum over a token's slots is a
// fixed butterfly (the same order on every run).
__device__ __forceinline__ void softmax_weights(int tb, int tend, int k,
                                                const float (*s_v)[kMaxK],
                                                float* __restrict__ w_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kp = (k <= 8) ? 8 : 16;
  const int tpw = 32 / kp;  // tokens per warp
  const int tl = warp * tpw + lane / kp, r = lane % kp;
  if (warp * tpw < kTokPerBlock) {
    const int tt = tb + tl;
    const bool on = tl < kTokPerBlock && tt < tend && r < k;
    const dflt ex = on ? df_softmax_term(s_v[tl][r], s_v[tl][0]) : dflt{0.0f, 0.0f};
    dflt den = ex;
    for (int off = kp >> 1; off > 0; off >>= 1) {
      const dflt o = {__shfl_xor_sync(0xffffffffu, den.hi, off),
                      __shfl_xor_sync(0xffffffffu, den.lo, off)};
      den = df_add(den, o);
    }
    if (on) w_out[(long long)tt * k + r] = df_div(ex, den).hi;
  }
}

// One warp per token, 32 tokens per block (one block = one row of the
// histogram): top-k of each token (topk_warp), then the block's weights and
// its per-expert counts hist[block][e].
template <int VPL>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float* __restrict__ part, int KS, int T, int E, int k, const float* __restrict__ bias,
    float* __restrict__ logits, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
    int32_t* __restrict__ hist, int* __restrict__ err) {
  __shared__ int cnt[kMaxE];
  __shared__ float s_v[kTokPerBlock][kMaxK];  // the kept logits of each token, in order
  const int warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kTokPerBlock + warp;
  if (t < T) topk_warp<VPL>(part, KS, T, E, k, bias, logits, idx_out, t, s_v[warp], cnt, err);
  __syncthreads();
  softmax_weights(blockIdx.x * kTokPerBlock, T, k, s_v, w_out);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[(long long)blockIdx.x * E + e] = cnt[e];
}

// Exclusive scan of one value per thread over the whole block (<= 1024
// threads); returns the thread's prefix and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
    if (lane == nw - 1) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Shared memory of offsets_and_tiles.
struct TileSmem {
  int warp_tot[32];
  int total;
  int clsb[17];
  int wcls[32][16];  // per warp: experts of each remainder class
};

// Offsets over the routed experts and the tile map, from every expert's
// count; one block, every thread (<= 1024, > E): thread e < E passes expert
// e's count, thread E the shared expert's (T; 0 without one), the others 0.
// Tile map: full kTileRows-row tiles first (expert order, shared last), then
// each expert's remainder tile, larger remainders first (ties in expert
// order).  The shared expert (index E, rows T*k .. T*k+T-1) takes part like
// any expert.
__device__ void offsets_and_tiles(int cnt, int T, int E, int k, int has_shared,
                                  int32_t* __restrict__ offsets, int4* __restrict__ tiles,
                                  int32_t* __restrict__ ntiles, TileSmem& sm) {
  const int tid = threadIdx.x;
  const int nexp = E + (has_shared ? 1 : 0);
  // offsets over the routed experts
  const int off = block_exclusive_scan(tid < E ? cnt : 0, sm.warp_tot, &sm.total);
  if (tid <= E) offsets[tid] = (tid < E) ? off : sm.total;
  // full tiles, all experts (shared last)
  const int nf = (tid < nexp) ? cnt / kTileRows : 0;
  const int full_off = block_exclusive_scan(nf, sm.warp_tot, &sm.total);
  const int total_full = sm.total;
  // remainder tiles: class c = npad/16 - 1, larger classes first
  static_assert(kTileRows / 16 <= 16, "remainder classes");
  const int tail = (tid < nexp) ? cnt % kTileRows : 0;
  const int cls = tail ? ((tail + 15) >> 4) - 1 : -1;
  if (tid < 17) sm.clsb[tid] = 0;
  if (tid < 32 * 16) (&sm.wcls[0][0])[tid] = 0;
  __syncthreads();
  if (cls >= 0) atomicAdd(&sm.clsb[cls], 1);
  // rank of the expert among the lower-indexed experts of its class: within
  // the warp by matching lanes, then the counts of the earlier warps
  const int lane = tid & 31, wid = tid >> 5;
  const unsigned same = __match_any_sync(0xffffffffu, cls);
  const int wrank = __popc(same & ((1u << lane) - 1u));
  if (cls >= 0 && wrank == 0) sm.wcls[wid][cls] = __popc(same);
  __syncthreads();
  if (tid == 0) {
    int run = total_full;
    for (int c = 15; c >= 0; --c) {
      const int n = sm.clsb[c];
      sm.clsb[c] = run;
      run += n;
    }
    *ntiles = run;
  }
  __syncthreads();
  if (tid < nexp) {
    const int e = tid;
    const int row_base = (e < E) ? off : T * k;
    for (int i = 0; i < nf; ++i)
      tiles[full_off + i] = make_int4(e, row_base + i * kTileRows, kTileRows, kTileRows);
    if (cls >= 0) {
      int rank = wrank;
      for (int w = 0; w < wid; ++w) rank += sm.wcls[w][cls];
      tiles[sm.clsb[cls] + rank] = make_int4(e, row_base + nf * kTileRows, tail, (tail + 15) & ~15);
    }
  }
}

// Single block.  Per expert: exclusive scan of the block histograms over
// blocks (base[b][e]), the total count, the exclusive scan over experts
// (offsets), and the tile map: full 256-row tiles first (expert order), then
// each expert's remainder tile, larger remainders first (ties in expert
// order).  The shared expert (index E, all T tokens, rows T*k..T*k+T-1)
// takes part like any expert.
// The scan over blocks is split by experts over the grid: block g takes
// experts [g*EB, (g+1)*EB) with P = 1024 / EB threads per expert (thread
// p*EB + e), each over a contiguous range of blocks, 16 loads in flight at a
// time; the ranges' sums are exchanged in shared memory, then each thread
// writes its range's bases from its range prefix.  The last block to finish
// (a ticket counter, reset by that block for the next call) computes the
// offsets and the tile map from every expert's count.
constexpr int kScanBatch = 16;
__global__ void __launch_bounds__(1024) scan_tiles_kernel(
    const int32_t* __restrict__ hist, int nblk, int T, int E, int k, int has_shared,
    int32_t* __restrict__ base, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int4* __restrict__ tiles, int32_t* __restrict__ ntiles, unsigned* __restrict__ ticket) {
  __shared__ TileSmem tsm;
  __shared__ int s_part[1024];
  __shared__ int s_last;
  const int tid = threadIdx.x;

  const int EB = (E + gridDim.x - 1) / gridDim.x;  // experts of this block
  const int e0 = blockIdx.x * EB, ne = min(E, e0 + EB) - e0;
  const int P = blockDim.x / EB;  // >= 2 (EB <= 512)
  const int pe = tid % EB, pp = tid / EB;
  const int ex = e0 + pe;
  const int nbp = (nblk + P - 1) / P;
  const int b0 = pp * nbp, b1 = min(nblk, b0 + nbp);
  const bool mine = pp < P && pe < ne;
  int part = 0;
  if (mine) {
    for (int b = b0; b < b1; b += kScanBatch) {
      int c[kScanBatch];
#pragma unroll
      for (int q = 0; q < kScanBatch; ++q)
        c[q] = (b + q < b1) ? hist[(long long)(b + q) * E + ex] : 0;
#pragma unroll
      for (int q = 0; q < kScanBatch; ++q) part += c[q];
    }
  }
  if (tid < P * EB) s_part[tid] = part;
  __syncthreads();
  if (mine) {
    int pre = 0, tot = 0;
    for (int q = 0; q < P; ++q) {
      const int v = s_part[q * EB + pe];
      pre += (q < pp) ? v : 0;
      tot += v;
    }
    int run = pre;
    for (int b = b0; b < b1; b += kScanBatch) {
      int c[kScanBatch];
#pragma unroll
      for (int q = 0; q < kScanBatch; ++q)
        c[q] = (b + q < b1) ? hist[(long long)(b + q) * E + ex] : 0;
#pragma unroll
      for (int q = 0; q < kScanBatch; ++q) {
        if (b + q < b1) base[(long long)(b + q) * E + ex] = run;
        run += c[q];
      }
    }
    if (pp == 0) counts[ex] = tot;
  }
  // the last block continues with every expert's count
  if (gridDim.x > 1) {
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  } else {
    __syncthreads();
  }
  int cnt = 0;
  if (tid < E) cnt = __ldcg(counts + tid);
  if (tid == E && has_shared) cnt = T;
  if (tid == 0 && gridDim.x > 1) *ticket = 0u;  // for the next call
  __syncthreads();
  offsets_and_tiles(cnt, T, E, k, has_shared, offsets, tiles, ntiles, tsm);
}

// Scatter (stable counting sort by (expert, token)).  Row of assignment
// (t, j) with expert e = offsets[e] + base[block][e] + (number of tokens
// of this block before t that chose e).  Also fills, per grouped row, the
// routing weight and the contribution row t*(k+has_shared)+j, and the rows of
// the shared expert (T*k + t; their weight, the gate, comes with the
// permuted activations).
__global__ void __launch_bounds__(256) scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ base, int T, int E, int k,
    int has_shared, int32_t* __restrict__ perm, int32_t* __restrict__ slot,
    int32_t* __restrict__ dst, float* __restrict__ wrow) {
  __shared__ uint32_t mask[kMaxE][kTokPerBlock / 32];
  const int b = blockIdx.x;
  const int t0 = b * kTokPerBlock;
  const int k1 = k + (has_shared ? 1 : 0);
  for (int i = threadIdx.x; i < E * (kTokPerBlock / 32); i += blockDim.x)
    (&mask[0][0])[i] = 0u;
  __syncthreads();
  for (int a = threadIdx.x; a < kTokPerBlock * k; a += blockDim.x) {
    const int tl = a / k;
    const int t = t0 + tl;
    if (t < T) {
      const int e = idx[(long long)t * k + (a - tl * k)];
      atomicOr(&mask[e][tl >> 5], 1u << (tl & 31));
    }
  }
  __syncthreads();
  for (int a = threadIdx.x; a < kTokPerBlock * k; a += blockDim.x) {
    const int tl = a / k;
    const int j = a - tl * k;
    const int t = t0 + tl;
    if (t < T) {
      const int e = idx[(long long)t * k + j];
      int rank = 0;
      for (int wd = 0; wd < (tl >> 5); ++wd) rank += __popc(mask[e][wd]);
      rank += __popc(mask[e][tl >> 5] & ((1u << (tl & 31)) - 1u));  // tokens before t
      const int row = offsets[e] + base[(long long)b * E + e] + rank;
      perm[row] = t;
      slot[(long long)t * k + j] = row;
      wrow[row] = w[(long long)t * k + j];
      dst[row] = t * k1 + j;
    }
  }
  if (has_shared) {
    for (int tl = threadIdx.x; tl < kTokPerBlock; tl += blockDim.x) {
      const int t = t0 + tl;
      if (t < T) {
        const int row = T * k + t;
        perm[row] = t;
        dst[row] = t * k1 + k;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fused routing: top-k + histogram, scan + tile map, scatter, and the fp16
// activations the gate/up GEMM gathers from, with the shared-expert gate, in one
// cooperative launch of G persistent blocks (one per SM at most).  Block b
// owns the contiguous tokens [b tpb, (b+1) tpb); its per-expert counts are
// row b of the histogram, so the block order is the token order and the
// counting sort stays stable (rows of an expert group in ascending token
// order).  The only grid-wide step is one barrier between the histogram and
// the scan.
constexpr int kRouteThreads = 1024;
constexpr uint64_t kGridWaitNs = 2000000000ull;  // 2 s

struct RouteParams {
  const float* part;  // router partial logits [KS][T][E] (KS = 1: given logits)
  int KS, T, E, k, has_shared, d;
  const float* bias;       // [E] or null
  const uint16_t* x;       // bf16 [T][d], or null: no permuted activations
  const uint16_t* w_sg;    // bf16 [d] shared-expert gate (has_shared)
  float* logits;           // [T][E]
  int32_t* idx;            // [T][k]
  float* w;                // [T][k]
  float* sigma;            // [T]
  int32_t* hist;           // [G][E]
  int32_t* counts;         // [E]
  int32_t* offsets;        // [E+1]
  int32_t* perm;           // [T(k+1)] grouped row -> token
  int32_t* slot;           // [T][k] -> grouped row
  int32_t* dst;            // [T(k+1)] grouped row -> contribution row
  float* wrow;             // [T(k+1)] grouped row -> routing weight / gate (times s^2)
  float* xrow;             // [T(k+1)] grouped row -> activation scale s of its token
  float* xtok;             // [T] activation scale s of each token
  int* xscaled;            // set when some token of the call has s != 1
  int4* tiles;
  int32_t* ntiles;
  uint16_t* xp;            // fp16 [T][d]
  unsigned* bar;           // [2] grid barrier: arrivals, generation
  int* err;
};

// Grid-wide barrier of a cooperative launch (every block resident), passed
// once per launch: a block adds its arrival to bar[0] without waiting for
// the result and polls the count until every block has arrived (one L2 round
// trip after the last arrival); bar[1] counts the blocks that have left, and
// the last of them zeroes both for the next launch.  Gives up after
// kGridWaitNs, setting MOE_DEVERR_GRID_TIMEOUT (the results are then wrong,
// but the kernel ends).
__device__ void route_grid_sync(unsigned* bar, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= gridDim.x) break;
      if ((n & 63u) == 0 && globaltimer_ns() - t0 > kGridWaitNs) {
        atomicOr(err, MOE_DEVERR_GRID_TIMEOUT);
        break;
      }
    }
    if (atomicAdd(bar + 1, 1u) == gridDim.x - 1) {  // every block has left the wait
      bar[0] = 0u;
      bar[1] = 0u;
    }
  }
  __syncthreads();
}

template <int VPL>
__global__ void __launch_bounds__(kRouteThreads, 1) route_kernel(const __grid_constant__ RouteParams p) {
  __shared__ int cnt[kMaxE];       // block histogram, then running ranks
  __shared__ int row0[kMaxE];      // offsets[e] + this block's base for e
  __shared__ uint32_t mask[kMaxE]; // tokens of a 32-token group choosing e
  __shared__ float s_v[kTokPerBlock][kMaxK];
  __shared__ TileSmem tsm;
  __shared__ int s_before[kRouteThreads];  // partial column sums of the histogram
  __shared__ int s_all[kRouteThreads];
  __shared__ int s_scaled;  // some token of this block has s != 1
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, E = p.E, k = p.k, G = gridDim.x, b = blockIdx.x;
  const int k1 = k + (p.has_shared ? 1 : 0);
  const int tpb = (T + G - 1) / G;
  const int t0 = min(T, b * tpb), t1 = min(T, t0 + tpb);

  // ---- 1. top-k of the block's tokens (one warp per token), weights, counts
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  if (tid == 0) s_scaled = 0;
  __syncthreads();
  for (int tb = t0; tb < t1; tb += kTokPerBlock) {
    const int t = tb + warp;
    if (warp < kTokPerBlock && t < t1) {
      if constexpr (VPL == 8)
        topk_warp8(p.part, p.KS, T, E, k, p.bias, p.logits, p.idx, t, s_v[warp], cnt, p.err);
      else
        topk_warp<VPL>(p.part, p.KS, T, E, k, p.bias, p.logits, p.idx, t, s_v[warp], cnt, p.err);
    }
    __syncthreads();
    softmax_weights(tb, t1, k, s_v, p.w);
    __syncthreads();
  }
  for (int e = tid; e < E; e += blockDim.x) p.hist[(long long)b * E + e] = cnt[e];
  if (b == 0 && tid == 0 && p.x) *p.xscaled = 0;  // set after the barrier

  // ---- 2. the fp16 copy of the activations, from which the gate/up GEMM
  // gathers its token rows (one warp per token), and the shared gate sigma =
  // sigmoid(w_sg . x) on the way; before the barrier, which does not order
  // it (it needs no routing), so that its loads overlap the barrier's wait.
  // fp16 holds less range than bf16, so each token's row is divided by a
  // power of two s first: s = 1 while the row's largest magnitude is in
  // [2^-6, 2^6) (the usual activations: the copy is exact up to fp16
  // rounding), else 2^(floor(log2 max) - 1), which brings the largest value
  // into [2, 4); log2 s is clamped to [-60, 60].  The gate/up epilogue and
  // the row weights of the down projection (times s^2, step 4) undo it
  // exactly.  One pass converts with s = 1 while finding the largest
  // magnitude; a token that needs another s is converted again.
  if (p.x) {
    // a lane's loads of a row are issued together, 4 at a time
    auto convert = [&](const uint4* xr, uint4* xo, float inv, float* amax, float* dot) {
      for (int c0 = lane; c0 < p.d / 8; c0 += 32 * 4) {
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (c0 + 32 * i < p.d / 8) raw[i] = __ldg(xr + c0 + 32 * i);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + 32 * i;
          if (c >= p.d / 8) break;
          const uint32_t wv[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
          uint32_t hv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(wv[q] << 16);
            const float hi = __uint_as_float(wv[q] & 0xFFFF0000u);
            if (amax) *amax = fmaxf(*amax, fmaxf(fabsf(lo), fabsf(hi)));
            const __half2 h2 = __floats2half2_rn(lo * inv, hi * inv);
            hv[q] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          xo[c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          if (dot && p.has_shared) {
            const uint4 sg = __ldg(reinterpret_cast<const uint4*>(p.w_sg) + c);
            const uint32_t sv[4] = {sg.x, sg.y, sg.z, sg.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              *dot = fmaf(__uint_as_float(wv[q] << 16), __uint_as_float(sv[q] << 16), *dot);
              *dot = fmaf(__uint_as_float(wv[q] & 0xFFFF0000u), __uint_as_float(sv[q] & 0xFFFF0000u),
                          *dot);
            }
          }
        }
      }
    };
    for (int t = t0 + warp; t < t1; t += kRouteThreads / 32) {
      const uint4* xr = reinterpret_cast<const uint4*>(p.x + (long long)t * p.d);
      uint4* xo = reinterpret_cast<uint4*>(p.xp + (long long)t * p.d);
      float dot = 0.0f, amax = 0.0f;
      convert(xr, xo, 1.0f, &amax, &dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      int ex = 0;  // log2 s
      if (amax > 0.0f && (amax < 0.015625f || amax >= 64.0f)) {
        ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 128;  // floor(log2 max) - 1
        ex = min(max(ex, -60), 60);
      }
      const float s_t = __int_as_float((127 + ex) << 23);
      const float inv = __int_as_float((127 - ex) << 23);
      if (lane == 0 && !(amax * inv < 65520.0f) && amax == amax) atomicOr(p.err, MOE_DEVERR_FP16_RANGE);
      if (ex != 0) {
        __syncwarp();  // the first pass's stores of this row are done (same lanes)
        convert(xr, xo, inv, nullptr, nullptr);
        if (lane == 0) s_scaled = 1;
      }
      if (lane == 0) p.xtok[t] = s_t;
      if (p.has_shared) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (lane == 0) {
          const float sg = 1.0f / (1.0f + expf(-dot));
          p.sigma[t] = sg;
          p.wrow[T * k + t] = sg * (s_t * s_t);
          p.xrow[T * k + t] = s_t;
        }
      }
    }
  }
  route_grid_sync(p.bar, p.err);
  if (tid == 0 && s_scaled) atomicOr(p.xscaled, 1);

  // ---- 3. per expert: this block's base (the counts of the blocks before
  // it) and the total.  Thread tid = part * E + e sums part `part` of the
  // blocks' counts of expert e (its loads issued together, kHistBatch at a
  // time); one thread per expert adds the parts in order.
  {
    constexpr int kHistBatch = 20;
    const int nparts = kRouteThreads / E;  // >= 2 (E <= kMaxE = 512)
    const int chunk = (G + nparts - 1) / nparts;
    const int part = tid / E, e = tid - part * E;
    if (part < nparts) {
      const int g0 = min(G, part * chunk), g1 = min(G, g0 + chunk);
      int before = 0, all = 0;
      for (int gb = g0; gb < g1; gb += kHistBatch) {
        int cv[kHistBatch];
#pragma unroll
        for (int i = 0; i < kHistBatch; ++i)
          cv[i] = (gb + i < g1) ? __ldcg(p.hist + (long long)(gb + i) * E + e) : 0;
#pragma unroll
        for (int i = 0; i < kHistBatch; ++i) {
          all += cv[i];
          before += (gb + i < b) ? cv[i] : 0;
        }
      }
      s_before[tid] = before;
      s_all[tid] = all;
    }
    __syncthreads();
  }
  int tot = 0, base = 0;
  if (tid < E) {
    const int nparts = kRouteThreads / E;
    for (int q = 0; q < nparts; ++q) {
      tot += s_all[q * E + tid];
      base += s_before[q * E + tid];
    }
  }
  // exclusive scan over the experts' totals
  const int off = block_exclusive_scan(tid < E ? tot : 0, tsm.warp_tot, &tsm.total);
  if (tid < E) {
    row0[tid] = off + base;
    cnt[tid] = 0;  // running ranks of step 4
    mask[tid] = 0u;
  }
  if (b == 0) {
    if (tid < E) p.counts[tid] = tot;
    int c = (tid < E) ? tot : 0;
    if (tid == E && p.has_shared) c = T;
    offsets_and_tiles(c, T, E, k, p.has_shared, p.offsets, p.tiles, p.ntiles, tsm);
  }
  __syncthreads();

  // ---- 4. scatter, 32 tokens at a time: row of (t, j) with expert e =
  // row0[e] + (tokens of this block before t that chose e); the row weight
  // carries s^2 of its token, the row's activation scale s
  for (int tb = t0; tb < t1; tb += 32) {
    for (int a = tid; a < 32 * k; a += blockDim.x) {
      const int tl = a / k, t = tb + tl;
      if (t < t1) atomicOr(&mask[p.idx[(long long)t * k + (a - tl * k)]], 1u << tl);
    }
    __syncthreads();
    for (int a = tid; a < 32 * k; a += blockDim.x) {
      const int tl = a / k, j = a - tl * k, t = tb + tl;
      if (t < t1) {
        const int e = p.idx[(long long)t * k + j];
        const int row = row0[e] + cnt[e] + __popc(mask[e] & ((1u << tl) - 1u));
        const float st = p.x ? p.xtok[t] : 1.0f;
        p.perm[row] = t;
        p.slot[(long long)t * k + j] = row;
        p.wrow[row] = p.w[(long long)t * k + j] * (st * st);
        if (p.x) p.xrow[row] = st;
        p.dst[row] = t * k1 + j;
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
      cnt[e] += __popc(mask[e]);
      mask[e] = 0u;
    }
    __syncthreads();
  }
  if (p.has_shared) {
    for (int t = t0 + tid; t < t1; t += blockDim.x) {
      p.perm[T * k + t] = t;
      p.dst[T * k + t] = t * k1 + k;
    }
  }
}

// out[t][f] = sum_{j=0}^{k1-1} Y[t*k1 + j][f], fp32 in slot order (the
// shared expert's term last), rounded once to bf16.  The routing weights were
// applied when the rows of Y were written.  A thread's loads of all k1 rows
// are issued before the sum.  K1 > 0: exactly K1 rows per token (registers
// for K1 loads only, so more blocks are resident); K1 = 0: any k1 up to
// kMaxK + 1.  Persistent blocks stride over the tokens (no partial last wave).
// A non-finite output (an intermediate beyond fp16's range on the way: the
// prefill path's H is fp16) sets MOE_DEVERR_FP16_RANGE.
template <int K1>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ Y, int k1,
                                                     int d, int T, uint16_t* __restrict__ out,
                                                     int* __restrict__ err) {
  constexpr int NR = K1 > 0 ? K1 : kMaxK + 1;
  const int nr = K1 > 0 ? K1 : k1;
  bool bad = false;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint4 rv[NR];
#pragma unroll
      for (int j = 0; j < NR; ++j)
        if (j < nr)
          rv[j] = __ldcs(reinterpret_cast<const uint4*>(Y + ((long long)t * nr + j) * d + c));
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        if (j >= nr) break;
        const uint4 raw = rv[j];
        const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] += __uint_as_float(v[q] << 16);
          acc[2 * q + 1] += __uint_as_float(v[q] & 0xFFFF0000u);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        o[q] = *reinterpret_cast<const uint32_t*>(&b2);
        bad |= !(fabsf(acc[2 * q]) <= 3.4e38f) || !(fabsf(acc[2 * q + 1]) <= 3.4e38f);
      }
      *reinterpret_cast<uint4*>(out + (long long)t * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (bad) atomicOr(err, MOE_DEVERR_FP16_RANGE);
}

// Blocks of the fused routing launch: one per 32 tokens, at most as many as
// can be resident at once (a cooperative launch; one per SM).
template <int VPL>
cudaError_t launch_route_vpl(const Handle* h, const RouteParams& p, cudaStream_t st) {
  static int per_sm = -1;
  if (per_sm < 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_kernel<VPL>, kRouteThreads,
                                                      0) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      return cudaErrorLaunchOutOfResources;
    }
  }
  const int want = (p.T + kTokPerBlock - 1) / kTokPerBlock;
  const int cap = h->num_sms * per_sm;
  const int G = want < cap ? want : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel<VPL>, p);
}

}  // namespace

cudaError_t launch_route(const Handle* h, const float* part, int KS, int T, const float* bias,
                         const uint16_t* x, cudaStream_t st) {
  const moe_config& c = h->cfg;
  const Workspace& ws = h->ws;
  RouteParams p{};
  p.part = part;
  p.KS = KS;
  p.T = T;
  p.E = c.E;
  p.k = c.k;
  p.has_shared = c.has_shared;
  p.d = c.d;
  p.bias = bias;
  p.x = x;
  p.w_sg = h->w_sg;
  p.logits = ws.logits;
  p.idx = ws.idx;
  p.w = ws.w;
  p.sigma = ws.sigma;
  p.hist = ws.hist;
  p.counts = ws.counts;
  p.offsets = ws.offsets;
  p.perm = ws.perm;
  p.slot = ws.slot;
  p.dst = ws.dst;
  p.wrow = ws.wrow;
  p.xrow = ws.xrow;
  p.xtok = ws.xtok;
  p.xscaled = reinterpret_cast<int*>(ws.ticket + 1);
  p.tiles = ws.tiles;
  p.ntiles = ws.ntiles;
  p.xp = ws.xp;
  p.bar = ws.ticket + 2;
  p.err = h->dev_err;
  return c.E <= 256 ? launch_route_vpl<8>(h, p, st) : launch_route_vpl<16>(h, p, st);
}

namespace {
// resident blocks of a combine variant (persistent grid)
template <int K1>
int combine_grid(const Handle* h, int threads, int T) {
  static int per_sm = -1;
  if (per_sm < 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<K1>, threads, 0) !=
            cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
  }
  const int cap = h->num_sms * per_sm;
  return T < cap ? T : cap;
}
}  // namespace

cudaError_t launch_combine(const Handle* h, int T, uint16_t* y, cudaStream_t st) {
  const moe_config& c = h->cfg;
  const int threads = c.d / 8 < 256 ? c.d / 8 : 256;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  if (k1 == 9)
    return launch_kernel(combine_kernel<9>, dim3(combine_grid<9>(h, threads, T)), dim3(threads), 0,
                         st, (const uint16_t*)h->ws.Y, k1, c.d, T, y, h->dev_err);
  return launch_kernel(combine_kernel<0>, dim3(combine_grid<0>(h, threads, T)), dim3(threads), 0,
                       st, (const uint16_t*)h->ws.Y, k1, c.d, T, y, h->dev_err);
}


// ---------------------------------------------------------------------------
// Routing from given logits with no device allocation.
//
// For callers that cannot call cudaMalloc: code running inside a device
// memory allocator or its callbacks, serving loops that must never hit
// cudaMalloc's implicit device synchronisation, and programs whose device
// memory is entirely owned by another framework.  The kernels' scratch lives
// in one file-scope device array of fixed size that every GPU loading this
// library holds until the process exits.
namespace {

constexpr int kNaMaxT = 2048;  // tokens per call
constexpr int kNaMaxE = 256;   // experts
constexpr int kNaMaxK = kMaxK; // kept experts per token
constexpr int kNaBlk = kNaMaxT / kTokPerBlock;
constexpr int kNaTiles = kNaMaxT * kNaMaxK / kTileRows + kNaMaxE + 2;

constexpr size_t na_align(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kNaLogits = 0;
constexpr size_t kNaHist = na_align(kNaLogits + sizeof(float) * kNaMaxT * kNaMaxE);
constexpr size_t kNaBase = na_align(kNaHist + sizeof(int32_t) * kNaBlk * kNaMaxE);
constexpr size_t kNaDst = na_align(kNaBase + sizeof(int32_t) * kNaBlk * kNaMaxE);
constexpr size_t kNaWrow = na_align(kNaDst + sizeof(int32_t) * kNaMaxT * kNaMaxK);
constexpr size_t kNaTilesOff = na_align(kNaWrow + sizeof(float) * kNaMaxT * kNaMaxK);
constexpr size_t kNaNtiles = na_align(kNaTilesOff + sizeof(int4) * kNaTiles);
constexpr size_t kNaErr = na_align(kNaNtiles + 16);
constexpr size_t kNaBytes = na_align(kNaErr + 16);  // about 2.5 MB

// The scratch.  Host code must not pass &g_na_scratch to a kernel: on the host
// the name is only a stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_na_scratch[kNaBytes];

std::mutex g_na_mutex;
unsigned char* g_na_ptr[64] = {};  // device address of g_na_scratch, per device

cudaError_t na_scratch(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_na_scratch);
    if (e != cudaSuccess) return e;
    g_na_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_na_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_route_from_logits_noalloc(const float* logits, int T, int E, int k,
                                                    const float* logit_bias, int32_t* idx,
                                                    float* w, int32_t* counts, int32_t* offsets,
                                                    int32_t* perm, int32_t* slot, void* stream) {
  using namespace moe;
  if (T < 0 || T > kNaMaxT || E < 1 || E > kNaMaxE || k < 1 || k > kNaMaxK || k > E)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w || !counts || !offsets || !perm || !slot) return MOE_ERR_INVALID_ARG;
  // the same alignment as the handle-based routing calls: 4-byte elements
  auto al4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  if (!al4(logits) || !al4(logit_bias) || !al4(idx) || !al4(w) || !al4(counts) ||
      !al4(offsets) || !al4(perm) || !al4(slot))
    return MOE_ERR_INVALID_ARG;
  unsigned char* s = nullptr;
  if (na_scratch(&s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nblk = (T + kTokPerBlock - 1) / kTokPerBlock;
  int32_t* hist = reinterpret_cast<int32_t*>(s + kNaHist);
  int32_t* base = reinterpret_cast<int32_t*>(s + kNaBase);
  int4* tiles = reinterpret_cast<int4*>(s + kNaTilesOff);
  int32_t* ntiles = reinterpret_cast<int32_t*>(s + kNaNtiles);
  float* lg = reinterpret_cast<float*>(s + kNaLogits);
  int* err = reinterpret_cast<int*>(s + kNaErr);
  int32_t* dst = reinterpret_cast<int32_t*>(s + kNaDst);
  float* wrow = reinterpret_cast<float*>(s + kNaWrow);
  // Every scratch word is written before it is read: nothing to clear.  Each
  // launch's own status is checked (an error left by an earlier, unrelated
  // launch is neither reported here nor cleared).
  auto cfg = [&](int grid, int threads) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(grid);
    c.blockDim = dim3(threads);
    c.stream = st;
    return c;
  };
  cudaLaunchConfig_t c1 = cfg(nblk, kTopkThreads);
  if (cudaLaunchKernelEx(&c1, topk_kernel<8>, logits, 1, T, E, k, logit_bias, lg, idx, w, hist,
                         err) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t c2 = cfg(1, 1024);
  if (cudaLaunchKernelEx(&c2, scan_tiles_kernel, (const int32_t*)hist, nblk, T, E, k, 0, base,
                         counts, offsets, tiles, ntiles, (unsigned*)nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaLaunchConfig_t c3 = cfg(nblk, 256);
  if (cudaLaunchKernelEx(&c3, scatter_kernel, (const int32_t*)idx, (const float*)w,
                         (const int32_t*)offsets, (const int32_t*)base, T, E, k, 0, perm, slot,
                         dst, wrow) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
