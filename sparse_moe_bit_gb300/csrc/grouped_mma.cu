// Grouped tensor-core GEMM for sm_103a: tcgen05.mma with TMEM accumulators,
// token-row operands staged in shared memory by the tensor memory accelerator
// (2-D tensor tiles multicast across a cluster), 4-bit weights dequantised
// tile by tile inside the pipeline.
//
// One work unit computes two 128-row weight tiles (A0, A1) against one token
// tile of up to 256 rows (B), over K in blocks of 64 (one quantisation group
// per block):
//   router : A = router rows e..e+255 (bf16), B = token rows of x (bf16),
//            out = fp32 partial logits of one K split.
//   gate/up: A0 = gate rows f..f+127, A1 = up rows f..f+127 of one expert
//            (dequantised to fp16), B = the expert's grouped token rows of x
//            (fp16, already permuted into grouped-row order); epilogue
//            H = silu(A0 x) * (A1 x) -> fp16.
//   down   : A = down rows f..f+127 (dequantised), B = the expert's rows of
//            H; epilogue Y[dst] = w_row * (A x) -> bf16, written to the
//            token's contribution row (deterministic combine later).
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Dequantize weights during matrix multiplication" (one small weight tile
// at a time is expanded to 16-bit in on-chip memory and multiplied with the
// routed activation rows; fp32 accumulation; the full matrix is never
// written out) and §"Match tile size to expert load" (tile shape from the
// expert's row count: the token dimension N of each tile is the expert's
// remaining row count rounded up to 16, at most 256).
//
// Warp roles (640 threads, one CTA per SM, persistent over the unit list):
//   warp 0       B producer (the warp's lanes issue the 16-row TMA tiles)
//                and, for the router, the A bulk copies
//   warp 1       lane 0 issues tcgen05.mma; the warp owns the TMEM allocation
//   warp 2       lane 0 issues the bulk copies of the code ring
//   warps 4..11  dequantise the weight codes from the ring into fp16 A tiles
//                (128-byte swizzled, K-major): gate/up one row per thread,
//                down half a row per thread
//   warps 12..19 epilogue: tcgen05.ld, activation / scaling, staging in
//                shared memory, 16-byte stores of 64-byte row segments
// Rings: A 2 stages, B 3 stages, codes 4 (gate/up) or 8 (down).  TMEM: two
// fp32 accumulators of 256 columns (gate/up and router: tiles A0 and A1 of
// one unit; down: two units in turn).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 640;
constexpr int kDeqWarps = 8;   // warps 4 .. 11
constexpr int kEpiWarp0 = 12;  // warps 12 .. 19
constexpr int kHalfChunk = 4608;  // 128 rows x (32 B codes + 4 B scale/bias)
constexpr int kAStages = 2;
constexpr int kBStage = 32768;   // up to 256 x 64 x 16-bit
constexpr int kEpiWarps = 8;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Per-mode shape of a work unit and of the pipeline:
//   NA   128-row weight tiles per unit (gate/up: the gate and the up tile of
//        the same features; router: 256 experts; down: 128 output rows, one
//        half of a 256-row code chunk)
//   NACC TMEM accumulator buffers: two fit when a unit needs only 256
//        columns (one tile), so that the down projection's epilogue (the
//        contribution rows, the largest write of the block) overlaps the
//        next unit's MMAs
//   CST  stages of the code ring: the codes and scale/bias words of a unit's
//        chunk (gate/up: 256 rows, 9 KB per K block) or half chunk (down:
//        4.5 KB) arrive by bulk copy, far enough ahead to hide the memory
//        latency that limited dequantisation from registers loaded three K
//        blocks ahead (cold experts at small T come from HBM)
template <int MODE>
struct Cfg {
  static constexpr int NA = (MODE == MMA_DOWN) ? 1 : 2;
  static constexpr int NACC = (MODE == MMA_DOWN) ? 2 : 1;
  static constexpr int NISS = NA;  // MMA-issuing threads (one per weight tile)
  static constexpr int CST = (MODE == MMA_DOWN) ? 8 : (MODE == MMA_GATEUP ? 4 : 0);
  static constexpr int CODE_STAGE = NA * kHalfChunk;
  static constexpr int B_STAGES = 3;
  static constexpr int A_STAGE = NA * 16384;
  // epilogue: per chunk of 16 rows, NSEG 64-byte segments per row (down: one
  // per weight tile; gate/up: one, the SwiGLU of the tile pair)
  static constexpr int NSEG = (MODE == MMA_DOWN) ? NA : 1;
  static constexpr int STAGE_BUF = 16 * 64 * NSEG;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kAStages * A_STAGE;
  static constexpr int OFF_CODE = OFF_B + B_STAGES * kBStage;
  static constexpr int OFF_STAGE = OFF_CODE + CST * CODE_STAGE;
  static constexpr int OFF_BAR = OFF_STAGE + kEpiWarps * 2 * STAGE_BUF;
  static constexpr int NUM_BARS = 2 * kAStages + 2 * B_STAGES + 2 * NACC + 2 * CST + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Unit {
  int expert, row0, nrows, npad, m, ks;
};

__device__ __forceinline__ Unit get_unit(const MmaParams& p, int mode, int u) {
  Unit o;
  const int tile = u / p.units_per_tile;
  const int r = u - tile * p.units_per_tile;
  if (mode == MMA_ROUTER) {
    o.ks = r / p.m_units;
    o.m = r - o.ks * p.m_units;
    o.expert = 0;
    o.row0 = tile * p.router_n;
    o.nrows = min(p.router_n, p.rows_total - o.row0);
  } else {
    const int4 t = p.tiles[tile];
    o.expert = t.x;
    o.row0 = t.y;
    o.nrows = t.z;
    o.ks = 0;
    o.m = r;
  }
  o.npad = (o.nrows + 15) & ~15;
  return o;
}

template <int MODE>
struct Smem {
  using C = Cfg<MODE>;
  uint32_t base;
  __device__ uint32_t a(int s) const { return base + C::OFF_A + s * C::A_STAGE; }
  __device__ uint32_t b(int s) const { return base + C::OFF_B + s * kBStage; }
  __device__ uint32_t stage(int w, int i) const {
    return base + C::OFF_STAGE + (w * 2 + i) * C::STAGE_BUF;
  }
  __device__ uint32_t bar(int i) const { return base + C::OFF_BAR + 8 * i; }
  __device__ uint32_t a_full(int s) const { return bar(s); }
  __device__ uint32_t a_empty(int s) const { return bar(kAStages + s); }
  __device__ uint32_t b_full(int s) const { return bar(2 * kAStages + s); }
  __device__ uint32_t b_empty(int s) const { return bar(2 * kAStages + C::B_STAGES + s); }
  __device__ uint32_t acc_full(int b) const { return bar(2 * kAStages + 2 * C::B_STAGES + b); }
  __device__ uint32_t acc_empty(int b) const {
    return bar(2 * kAStages + 2 * C::B_STAGES + C::NACC + b);
  }
  __device__ uint32_t code(int s) const { return base + C::OFF_CODE + s * C::CODE_STAGE; }
  __device__ uint32_t c_full(int s) const {
    return bar(2 * kAStages + 2 * C::B_STAGES + 2 * C::NACC + s);
  }
  __device__ uint32_t c_empty(int s) const {
    return bar(2 * kAStages + 2 * C::B_STAGES + 2 * C::NACC + C::CST + s);
  }
  __device__ uint32_t drain() const { return bar(C::NUM_BARS - 1); }
};

__device__ __forceinline__ void record_timeout(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  atomicOr(err, MOE_DEVERR_WAIT_TIMEOUT);
}

// mbarrier wait that suspends the thread in hardware between checks
__device__ __forceinline__ bool try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            int* err) {
  if (try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (try_wait_sleep(bar, parity)) return true;
    if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
      record_timeout(abort_flag, err);
      return false;
    }
  }
}

// every lane waits (suspended); the give-up decision is the warp's together
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err) {
  bool ok = try_wait_sleep(bar, parity);
  if (__all_sync(0xffffffffu, ok)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    ok = ok || try_wait_sleep(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    int bail = 0;
    if ((threadIdx.x & 31) == 0) bail = (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs);
    if (__shfl_sync(0xffffffffu, bail, 0)) {
      if ((threadIdx.x & 31) == 0) record_timeout(abort_flag, err);
      return false;
    }
  }
}

// The four fp16 pairs s*q + beta of the 8 codes of word v (pair j = K
// indices 2j, 2j+1 in the nibbles at bits 4j and 16+4j).  A nibble ORed
// into the low mantissa bits of 1024.0 (ulp 1) gives 1024 + q; the nibble
// at bits 4..7 ORed into 64.0 (ulp 1/16) gives 64 + q: so pairs 0 and 1
// need no shift and pairs 2 and 3 one 8-bit shift of the word.  One
// subtraction makes q exact, one fused multiply-add rounds s*q + beta once.
__device__ __forceinline__ uint4 dequant_word(uint32_t v, uint32_t s2, uint32_t b2) {
  const uint32_t v8 = v >> 8;
  const uint32_t t[4] = {(v & 0x000F000Fu) | 0x64006400u, (v & 0x00F000F0u) | 0x54005400u,
                         (v8 & 0x000F000Fu) | 0x64006400u, (v8 & 0x00F000F0u) | 0x54005400u};
  const __half2 m1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
  const __half2 m64 = __halves2half2(__ushort_as_half(0x5400), __ushort_as_half(0x5400));
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&t[j]), (j & 1) ? m64 : m1024);
    const __half2 h = __hfma2(q, *reinterpret_cast<const __half2*>(&s2),
                              *reinterpret_cast<const __half2*>(&b2));
    r[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// TMA load of B: a 2-D tile (16 rows).  With CL > 1 the data is multicast to
// the same shared-memory offset of every CTA of the cluster and each CTA's
// barrier at `bar` receives its bytes.
template <int CL>
__device__ __forceinline__ void tma_tile_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  if (CL == 1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(bar)
        : "memory");
  } else {
    const uint16_t mask = (uint16_t)((1u << CL) - 1u);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(bar), "h"(mask)
        : "memory");
  }
}

// tcgen05 commit that arrives on `bar` in every CTA of the cluster
template <int CL>
__device__ __forceinline__ void tc_commit_cluster(uint32_t bar) {
  if (CL == 1) {
    tc_commit(bar);
  } else {
    const uint16_t mask = (uint16_t)((1u << CL) - 1u);
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  }
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// CL: CTAs per cluster.  The CL CTAs of a cluster work on the same token tile
// (consecutive weight units m), each fetching every CL-th 16-row slab of B and
// multicasting it to all of them; a B slot is reused only after every CTA's
// MMAs have read it (each MMA commit arrives on the slot's barrier in all CTAs).
template <int MODE, int CL>
__global__ void __launch_bounds__(kThreads, 1) grouped_mma_kernel(const __grid_constant__ MmaParams p) {
  using C = Cfg<MODE>;
  constexpr int kBStages = C::B_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem<MODE> S{smem_u32(smem)};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nunits =
      (MODE == MMA_ROUTER) ? p.nunits_host : (*p.ntiles_dev) * p.units_per_tile;
  // work: the i-th cluster unit of cluster cid is cunit(i), snake order over
  // the tile list (sorted by size: full tiles first, then remainders largest
  // first), so that every cluster gets a similar mix; the CTA of rank r takes
  // unit cu * CL + r (same tile for the whole cluster, weight unit m =
  // consecutive)
  const int ncu = nunits / CL;
  const int cid = (CL == 1) ? (int)blockIdx.x : (int)cluster_id();
  const int ncl = (CL == 1) ? (int)gridDim.x : (int)cluster_count();
  const int crank = (CL == 1) ? 0 : (int)cluster_rank();
  if (cid >= ncu) return;  // uniform over the cluster
  auto cunit = [&](int i) {
    const int base = i * ncl;
    return (i & 1) ? base + (ncl - 1 - cid) : base + cid;
  };
  const int nmy = ncu / ncl + ((cunit(ncu / ncl) < ncu) ? 1 : 0);  // this cluster's units

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(S.a_full(s), MODE == MMA_ROUTER ? 1 : kDeqWarps);
      mbar_init(S.a_empty(s), C::NISS);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(S.b_full(s), 1);
      mbar_init(S.b_empty(s), CL * C::NISS);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(S.acc_full(b), C::NISS);
      mbar_init(S.acc_empty(b), kEpiWarps);
    }
    for (int s = 0; s < C::CST; ++s) {
      mbar_init(S.c_full(s), 1);
      mbar_init(S.c_empty(s), kDeqWarps);
    }
    mbar_init(S.drain(), C::NISS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // peers' barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kbu = p.kb_per_unit;

  if (warp == 0) {
    // ------------------------------------------------------ B (+ router A)
    uint32_t gb = 0, ga = 0;
    bool ok = true;
    Unit tn = get_unit(p, MODE, cunit(0) * CL + crank);
    for (int i = 0; i < nmy && ok; ++i) {
      const Unit t = tn;
      if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank);
      const int k0 = t.ks * kbu;
      const uint8_t* asrc = p.wA + (long long)t.m * p.a_unit_stride + (long long)k0 * p.a_chunk;
      for (int kb = 0; kb < kbu; ++kb) {
        if (MODE == MMA_ROUTER) {
          const int s = ga % kAStages;
          if (!warp_wait(S.a_empty(s), ((ga / kAStages) & 1) ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(S.a_full(s), kRouterChunk);
            bulk_g2s(S.a(s), asrc + (long long)kb * p.a_chunk, kRouterChunk, S.a_full(s));
          }
          ++ga;
        }
        const int s = gb % kBStages;
        if (!warp_wait(S.b_empty(s), ((gb / kBStages) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t bs = S.b(s);
        const int x = (k0 + kb) * 64;
        // the whole tile arrives in every CTA; this CTA fetches 16-row slabs
        // crank, crank + CL, ... (one 2-D tile per slab)
        if (lane == 0) mbar_arrive_expect_tx(S.b_full(s), (uint32_t)t.npad * 128);
        __syncwarp();
        const int nslab = t.npad >> 4;
        for (int sl = crank + CL * lane; sl < nslab; sl += 32 * CL)
          tma_tile_2d<CL>(bs + sl * 2048, &p.tmB, x, t.row0 + 16 * sl, S.b_full(s));
        ++gb;
      }
    }
  } else if (warp == 1 || (warp == 3 && C::NISS == 2)) {
    // ---------------------------------------------------------- MMA issuer
    // With two weight tiles per unit, lane 0 of warp 1 issues tile 0's MMAs
    // and lane 0 of warp 3 tile 1's: a single thread issues a tcgen05.mma
    // no faster than one per ~56 cycles (measured), which bounded the small
    // tiles; two issuers on separate accumulators overlap.
    if (lane == 0) {
      const int q = (warp == 1) ? 0 : 1;  // this issuer's tile (two-tile units)
      uint32_t sa = 0, pa = 0, sb = 0, pb = 0;  // ring slots and phase parities
      Unit tn = get_unit(p, MODE, cunit(0) * CL + crank);
      for (int i = 0; i < nmy; ++i) {
        const Unit t = tn;  // the next unit's descriptor loads during this one
        if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank);
        const int ab = (C::NACC == 2) ? (int)(i & 1) : 0;
        const uint32_t aph = ((C::NACC == 2) ? (i >> 1) : i) & 1;
        if (!thread_wait(S.acc_empty(ab), aph ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(128, t.npad, MODE == MMA_ROUTER ? 1 : 0);
        bool ok = true;
        for (int kb = 0; kb < kbu; ++kb) {
          if (!thread_wait(S.a_full(sa), pa, abort_flag, p.err) ||
              !thread_wait(S.b_full(sb), pb, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K step kk: both operands advance by 32 bytes (2 in the
          // descriptor's address field, which holds the address / 16)
          const uint64_t bd = sdesc_k_sw128(S.b(sb));
#pragma unroll
          for (int j = 0; j < C::NA; ++j) {
            if (C::NISS == 2 && j != q) continue;
            const uint64_t ad = sdesc_k_sw128(S.a(sa) + j * 16384);
            // NA == 2: tile j -> columns 256 j; NACC == 2: buffer ab -> columns 256 ab
            const uint32_t dcol = tmem + 256 * (C::NA == 2 ? j : ab);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f16(dcol, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          }
          tc_commit(S.a_empty(sa));
          tc_commit_cluster<CL>(S.b_empty(sb));
          if (++sa == kAStages) { sa = 0; pa ^= 1; }
          if (++sb == (uint32_t)kBStages) { sb = 0; pb ^= 1; }
        }
        if (!ok) break;
        tc_commit(S.acc_full(ab));
      }
      // every issued MMA has finished before TMEM is released
      tc_commit(S.drain());
      mbar_wait_bounded(S.drain(), 0, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 2 && MODE != MMA_ROUTER) {
    // ------------------------------------------------ code ring
    if (lane == 0) {
      const int total = nmy * kbu;
      for (int g = 0; g < total; ++g) {
        constexpr int kCst = C::CST > 0 ? C::CST : 1;
        const int s = g % kCst;
        if (!thread_wait(S.c_empty(s), ((g / kCst) & 1) ^ 1, abort_flag, p.err)) break;
        const int j = g / kbu;
        const Unit u = get_unit(p, MODE, cunit(j) * CL + crank);
        if (C::NA == 2) {  // the whole chunk of unit m
          const uint8_t* ch = p.wA + (long long)u.expert * p.a_expert_stride +
                              (long long)u.m * p.a_unit_stride +
                              (long long)(g - j * kbu) * p.a_chunk;
          mbar_arrive_expect_tx(S.c_full(s), kCodeChunk);
          bulk_g2s(S.code(s), ch, kCodeChunk, S.c_full(s));
        } else {  // rows 128 (m % 2) .. +127 of chunk unit m / 2: codes, s,b words
          const uint8_t* ch = p.wA + (long long)u.expert * p.a_expert_stride +
                              (long long)(u.m >> 1) * p.a_unit_stride +
                              (long long)(g - j * kbu) * p.a_chunk;
          const int h = u.m & 1;
          mbar_arrive_expect_tx(S.c_full(s), kHalfChunk);
          bulk_g2s(S.code(s), ch + h * 4096, 4096, S.c_full(s));
          bulk_g2s(S.code(s) + 4096, ch + 8192 + h * 512, 512, S.c_full(s));
        }
      }
    }
  } else if (warp >= 4 && warp < 4 + kDeqWarps) {
    // ------------------------------------------------ dequantise
    if (MODE != MMA_ROUTER) {
      const int t = threadIdx.x - 128;  // 0..255
      // two tiles: row t of the unit (tile t >> 7); one tile: row t & 127,
      // K half t >> 7 (32 values)
      const int row = (C::NA == 2) ? t : (t & 127);
      const int kh = (C::NA == 2) ? 0 : (t >> 7);
      const int total = nmy * kbu;
      struct Codes {
        uint4 a0, a1;
        uint32_t sa;
      };
      // words w[i] (K 8 (4 kh + i) .. +7) of row r -> swizzled 16-byte chunks
      auto emit = [&](uint32_t a, int r, const Codes& cc) {
        const uint32_t s2 = __byte_perm(cc.sa, 0, 0x1010);
        const uint32_t b2 = __byte_perm(cc.sa, 0, 0x3232);
        const uint32_t rowb = a + (r >> 7) * 16384 + (r & 127) * 128;
        const uint32_t w[8] = {cc.a0.x, cc.a0.y, cc.a0.z, cc.a0.w,
                               cc.a1.x, cc.a1.y, cc.a1.z, cc.a1.w};
        constexpr int NW = (C::NA == 2) ? 8 : 4;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          const int c = 4 * kh + i;
          const uint4 d4 = dequant_word(w[i], s2, b2);
          st_shared_v4(rowb + ((c ^ (r & 7)) << 4), d4.x, d4.y, d4.z, d4.w);
        }
      };
      constexpr int kCst = C::CST > 0 ? C::CST : 1;
      for (int g = 0; g < total; ++g) {
        const int sc = g % kCst, sa = g % kAStages;
        if (!warp_wait(S.c_full(sc), (g / kCst) & 1, abort_flag, p.err) ||
            !warp_wait(S.a_empty(sa), ((g / kAStages) & 1) ^ 1, abort_flag, p.err))
          break;
        Codes cur;  // row `row` of the ring stage: codes, then the s,b word
        cur.a0 = ld_shared_v4(S.code(sc) + row * 32 + kh * 16);
        cur.a1 = (C::NA == 2) ? ld_shared_v4(S.code(sc) + row * 32 + 16) : cur.a0;
        cur.sa = ld_shared_u32(S.code(sc) + 32 * 128 * C::NA + row * 4);
        emit(S.a(sa), row, cur);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(S.c_empty(sc));
          mbar_arrive(S.a_full(sa));
        }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------- epilogue
    const int e = warp - kEpiWarp0;    // 0..7
    const int q = warp & 3;            // TMEM lane quarter
    const int half = e >> 2;           // columns [128*half, 128*half + 128)
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t nst = 0;
    Unit tn = get_unit(p, MODE, cunit(0) * CL + crank);
    for (int i = 0; i < nmy; ++i) {
      const Unit t = tn;
      if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank);
      const int c0 = half * 128;
      const int c1 = min(c0 + 128, t.npad);
      // row data of the warp's 128 columns, fetched while the MMAs run:
      // lane l holds rows c0 + l + 32 v, v = 0..3
      float rsc4[4] = {0.f, 0.f, 0.f, 0.f};
      int rdst4[4] = {0, 0, 0, 0};
      if (MODE == MMA_DOWN) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int n = c0 + lane + 32 * v;
          if (n < t.nrows) {
            rsc4[v] = p.row_scale[t.row0 + n];
            rdst4[v] = p.dst_row[t.row0 + n];
          }
        }
      }
      const int ab = (C::NACC == 2) ? (int)(i & 1) : 0;
      const uint32_t aph = ((C::NACC == 2) ? (i >> 1) : i) & 1;
      if (!warp_wait(S.acc_full(ab), aph, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + 256 * ab;
      for (int n0 = c0; n0 < c1; n0 += 16) {
        uint32_t r0[16], r1[16];
        tmem_ld16(tacc + n0, r0);
        if (C::NA == 2) tmem_ld16(tacc + 256 + n0, r1);
        const int nvalid = min(16, t.nrows - n0);
        // this chunk's rows n0..n0+15 are held by lanes (n0 - c0) % 32 + j
        // in register slot (n0 - c0) / 32
        const int vsel = (n0 - c0) >> 5;
        const int lsel = (n0 - c0) & 31;
        float rsc_v = rsc4[0];
        int rdst_v = rdst4[0];
#pragma unroll
        for (int v = 1; v < 4; ++v) {
          if (vsel == v) {
            rsc_v = rsc4[v];
            rdst_v = rdst4[v];
          }
        }
        const float rsc = __shfl_sync(0xffffffffu, rsc_v, (lsel + lane) & 31);
        const long long rdst = __shfl_sync(0xffffffffu, rdst_v, (lsel + lane) & 31);
        tmem_ld_wait();
        if (MODE == MMA_ROUTER) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j >= nvalid) break;
            const int row = t.row0 + n0 + j;
            const int ex = t.m * 256 + q * 32 + lane;
            float* o = p.out_f32 + ((long long)t.ks * p.rows_total + row) * p.E;
            if (ex < p.E) o[ex] = __uint_as_float(r0[j]);
            if (ex + 128 < p.E) o[ex + 128] = __uint_as_float(r1[j]);
          }
          continue;
        }
        // stage [16 rows][NSEG x 32 values] in shared memory, then 16-byte
        // vector stores of whole 64-byte row segments
        constexpr int NSEG = C::NSEG;
        const uint32_t sbuf = S.stage(e, nst & 1);
        __syncwarp();  // the buffer's previous reads are done
        if (nvalid > 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float v0 = __uint_as_float(r0[j]);
            if (MODE == MMA_GATEUP) {
              const float v1 = __uint_as_float(r1[j]);
              const float h = __fdividef(v0, 1.0f + __expf(-v0)) * v1;
              st_shared_u16(sbuf + j * 64 + lane * 2, __half_as_ushort(__float2half_rn(h)));
            } else {
              const float sc = __shfl_sync(0xffffffffu, rsc, j);
              st_shared_u16(sbuf + j * 64 * NSEG + lane * 2,
                            __bfloat16_as_ushort(__float2bfloat16_rn(sc * v0)));
              if (NSEG == 2)
                st_shared_u16(sbuf + j * 128 + 64 + lane * 2,
                              __bfloat16_as_ushort(__float2bfloat16_rn(sc * __uint_as_float(r1[j]))));
            }
          }
        }
        __syncwarp();
        // 16 rows x NSEG segments x four 16-byte pieces: piece pi = lane + 32 it
#pragma unroll
        for (int it = 0; it < 2 * NSEG; ++it) {
          const int pi = lane + 32 * it;
          const int j = pi / (4 * NSEG);
          const int seg = (pi >> 2) % NSEG;
          const int part = pi & 3;
          if (MODE == MMA_GATEUP) {
            if (j < nvalid) {
              const uint4 v = ld_shared_v4(sbuf + j * 64 + part * 16);
              const long long row = t.row0 + n0 + j;
              *reinterpret_cast<uint4*>(p.H + row * p.ldh + t.m * 128 + q * 32 + part * 8) = v;
            }
          } else {
            const long long dj = __shfl_sync(0xffffffffu, rdst, j);
            if (j < nvalid) {
              const uint4 v = ld_shared_v4(sbuf + j * 64 * NSEG + seg * 64 + part * 16);
              uint16_t* yr = p.Y + dj * p.ldy + t.m * (128 * NSEG) + seg * 128 + q * 32 + part * 8;
              *reinterpret_cast<uint4*>(yr) = v;
            }
          }
        }
        ++nst;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(S.acc_empty(ab));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // no CTA leaves while peers may still write to it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE, int CL>
cudaError_t launch_mode(const MmaParams& p, int grid, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_mma_kernel<MODE, CL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MODE>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // no more clusters than can be resident at once (persistent CTAs)
  static int max_grid = -1;
  if (max_grid < 0) {
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(CL);
    q.blockDim = dim3(kThreads);
    q.dynamicSmemBytes = Cfg<MODE>::SMEM;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = CL;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    q.attrs = a;
    q.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, grouped_mma_kernel<MODE, CL>, &q) != cudaSuccess ||
        ncl <= 0) {
      cudaGetLastError();
      ncl = 0;
    }
    max_grid = ncl * CL;
  }
  if (max_grid > 0 && grid > max_grid) grid = max_grid;
  grid = grid / CL * CL;
  if (grid < CL) grid = CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<MODE>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_mma_kernel<MODE, CL>, p);
}

// CTAs per cluster for a grouped launch: a power of two dividing the units
// of one tile.  Defaults measured on GB300 (T=4096, Zipf): gate/up 4, down 2;
// MOE_GEMM_CLUSTER (1, 2, 4) overrides both for tuning.
int cluster_for(int mode, int units_per_tile) {
  static int env = -1;
  if (env < 0) {
    const char* e = getenv("MOE_GEMM_CLUSTER");
    env = e ? atoi(e) : 0;
    if (env != 1 && env != 2 && env != 4) env = 0;
  }
  int cl = env ? env : (mode == MMA_GATEUP ? 4 : 2);
  while (cl > 1 && units_per_tile % cl != 0) cl >>= 1;
  return cl;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

}  // namespace

cudaError_t make_tmap_16bit(CUtensorMap* map, const void* base, long long rows, long long cols,
                            int box_rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_grouped_mma(int mode, const MmaParams& p, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  if (mode == MMA_ROUTER) return launch_mode<MMA_ROUTER, 1>(p, grid, st);
  const int cl = cluster_for(mode, p.units_per_tile);
  if (mode == MMA_GATEUP) {
    if (cl == 4) return launch_mode<MMA_GATEUP, 4>(p, grid, st);
    if (cl == 2) return launch_mode<MMA_GATEUP, 2>(p, grid, st);
    return launch_mode<MMA_GATEUP, 1>(p, grid, st);
  }
  if (cl == 4) return launch_mode<MMA_DOWN, 4>(p, grid, st);
  if (cl == 2) return launch_mode<MMA_DOWN, 2>(p, grid, st);
  return launch_mode<MMA_DOWN, 1>(p, grid, st);
}

}  // namespace moe
