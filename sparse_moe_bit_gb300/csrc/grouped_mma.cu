// Grouped tensor-core GEMM for sm_103a: tcgen05.mma with TMEM accumulators,
// 4-bit weights dequantised tile by tile inside the pipeline, token rows
// staged in shared memory.
//
// A work unit computes one or two 128-row weight tiles against one token
// tile of up to 192 rows (B), over K in blocks of 64 (one quantisation group
// per block):
//   router : A0, A1 = router rows e..e+255 (bf16, pre-swizzled, by bulk copy
//            into shared memory), B = token rows of x (bf16, 2-D TMA tiles),
//            out = fp32 partial logits of one K split.
//   gate/up: A0 = gate rows f..f+127, A1 = up rows f..f+127 of one expert
//            (dequantised to fp16 straight into TMEM), B = the tile's tokens
//            gathered through perm from the fp16 copy of x (cp.async);
//            epilogue H = silu(A0 x) * (A1 x) -> fp16.
//   down   : A = down rows f..f+127 (dequantised into TMEM), B = the
//            expert's rows of H (2-D TMA tiles), two K blocks per stage;
//            epilogue Y[dst] = w_row * (A x) -> bf16, written to the token's
//            contribution row (deterministic combine later).
// Gate/up and down run as CTA pairs (tcgen05 cta_group::2): the even CTA of
// a cluster of two issues M = 256 MMAs over both CTAs' A tiles (consecutive
// weight units) and each CTA holds half of the token tile.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Dequantize weights during matrix multiplication" (one small weight tile
// at a time is expanded to 16-bit on chip and multiplied with the routed
// activation rows; fp32 accumulation; the full matrix is never written out)
// and §"Match tile size to expert load" (tile shape from the expert's row
// count: the token dimension N of each tile is the expert's remaining row
// count rounded up to 16 (32 for pairs), at most 192).
//
// Warp roles (640 threads, one CTA per SM, persistent over the unit list):
//   warp 0       B producer (TMA tiles, or the gate/up row gather) and, for
//                the router, the A bulk copies
//   warp 1       issues tcgen05.mma (the whole warp runs the loop, one
//                elected lane issues; in a pair, the even CTA's) and owns the
//                TMEM allocation
//   warp 2       lane 0 issues the bulk copies of the code ring
//   warps 4..11  dequantise the weight codes from the ring into fp16 A tiles
//                in TMEM (gate/up one row per thread, every other K block;
//                down half a row per thread)
//   warps 12..19 epilogue: tcgen05.ld, activation / scaling, staging in
//                shared memory, 16-byte stores of 64-byte row segments (and,
//                in gate/up, the odd K blocks' dequantisation)
// TMEM (512 columns): gate/up two 192-column accumulators (gate, up) and a
// 2-stage A ring; down two 192-column accumulator buffers (the epilogue of a
// unit overlaps the next one's MMAs) and a 2-stage A ring of two K blocks;
// router two 128-column accumulators (token tiles of at most 128 rows) and
// 4-stage A and B rings.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <type_traits>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 640;
constexpr int kDeqWarps = 8;   // warps 4 .. 11
constexpr int kEpiWarp0 = 12;  // warps 12 .. 19
constexpr int kHalfChunk = 4608;  // 128 rows x (32 B codes + 4 B scale/bias)
constexpr int kEpiWarps = 8;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Per-mode shape of a work unit and of the pipeline:
//   NA     128-row weight tiles per unit (gate/up: the gate and the up tile
//          of the same features; router: 256 experts; down: 128 output
//          rows, one half of a 256-row code chunk)
//   NACC   TMEM accumulator buffers: two when a unit needs one tile, so that
//          the down projection's epilogue (the contribution rows, the
//          largest write of the block) overlaps the next unit's MMAs
//   NMAX   TMEM columns of one accumulator (the widest token tile)
//   TMEM_A the dequantised weight tile (the MMA's A operand) is written by
//          the dequantising threads straight into tensor memory (128 lanes x
//          32 columns per tile and K block, two fp16 per column), so that it
//          neither passes through shared memory nor is read from it by the
//          tensor core: shared-memory bandwidth, not the MMA rate, bounded
//          both grouped GEMMs with the A tiles in shared memory.  The TMEM
//          budget (512 columns) then holds the accumulators for token tiles
//          of up to 192 rows plus A_STAGES A stages.  The router's bf16 A
//          arrives pre-swizzled by bulk copy and stays in shared memory.
//   CST    stages of the code ring: the codes and scale/bias words of a
//          unit's chunk (gate/up: 256 rows, 9 KB per K block) or half chunk
//          (down: 4.5 KB) arrive by bulk copy, far enough ahead to hide the
//          memory latency (cold experts at small T come from HBM)
template <int MODE, bool PAIR>
struct Cfg {
  static constexpr bool TMEM_A = MODE != MMA_ROUTER;
  static constexpr int NA = (MODE == MMA_DOWN) ? 1 : 2;
  static constexpr int NACC = (MODE == MMA_DOWN) ? 2 : 1;
  // MMA-issuing warps: one.  (One per weight tile, on separate
  // accumulators, was 1 % slower for gate/up once each warp issued warp-wide.)
  static constexpr int NISS = 1;
  static constexpr int NMAX = TMEM_A ? kTileRows : 128;  // router token tiles: <= 128 rows
  // KPS: 64-wide K blocks per pipeline stage.  The down projection (one
  // weight tile, 4 MMAs per K block, one issuing thread) was bound by the
  // issuer's per-stage work (two barrier tests, a commit); two K blocks per
  // stage halve it.
  static constexpr int KPS = (MODE == MMA_DOWN) ? 2 : 1;
  static constexpr int A_COLS = NA * 32 * KPS;  // TMEM columns of one A stage
  static constexpr int A_COL0 = NMAX * (NA == 2 ? 2 : NACC);
  // as many A stages as the rest of TMEM holds (at most 8): the ring's depth
  // bounds the pipeline, whose round trip (dequantise, signal, MMA, commit)
  // is longer than one K block's MMAs
  static constexpr int A_STAGES =
      TMEM_A ? ((512 - A_COL0) / A_COLS < 8 ? (512 - A_COL0) / A_COLS : 8) : 4;
  static_assert(!TMEM_A || A_COL0 + A_STAGES * A_COLS <= 512, "TMEM budget");
  static_assert(TMEM_A || NA * NMAX <= 512, "TMEM budget");
  static constexpr int CST = (MODE == MMA_DOWN) ? 4 : (MODE == MMA_GATEUP ? 6 : 0);
  static constexpr int CODE_KB = NA * kHalfChunk;  // code bytes of one K block
  static constexpr int CODE_STAGE = CODE_KB * KPS;
  // B ring: up to NMAX token rows (a pair's CTA holds half of them) x 64 K
  // per K block (B_SUB bytes), KPS K blocks per stage
  static constexpr int B_STAGES =
      PAIR ? (KPS == 2 ? 4 : 8) : (MODE == MMA_GATEUP ? 6 : (MODE == MMA_ROUTER ? 4 : 3));
  static constexpr int B_SUB = (PAIR ? NMAX / 2 : NMAX) * 128;
  static constexpr int B_STAGE = B_SUB * KPS;
  static constexpr int A_STAGE = TMEM_A ? 0 : NA * 16384;  // shared-memory A (router)
  // epilogue: per chunk of 16 rows, NSEG 64-byte segments per row (down: one
  // per weight tile; gate/up: one, the SwiGLU of the tile pair)
  static constexpr int NSEG = (MODE == MMA_DOWN) ? NA : 1;
  static constexpr int STAGE_BUF = 16 * 64 * NSEG;
  // columns of the accumulator taken by each of the two epilogue halves
  static constexpr int EPI_COLS = NMAX / 2;
  static_assert(EPI_COLS % 16 == 0 && EPI_COLS <= 128, "epilogue column split");
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + A_STAGES * A_STAGE;
  static constexpr int OFF_CODE = OFF_B + B_STAGES * B_STAGE;
  static constexpr int OFF_STAGE = OFF_CODE + CST * CODE_STAGE;
  static constexpr int OFF_BAR = OFF_STAGE + kEpiWarps * 2 * STAGE_BUF;
  static constexpr int NUM_BARS = 2 * A_STAGES + 2 * B_STAGES + 2 * NACC + 2 * CST + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Unit {
  int expert, row0, nrows, npad, m, ks;
};

// pad: token rows per MMA column step of the tile (16; 32 for CTA pairs, whose
// two halves of B must each be whole 16-row slabs)
__device__ __forceinline__ Unit get_unit(const MmaParams& p, int mode, int u, int pad) {
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
  o.npad = (o.nrows + pad - 1) & ~(pad - 1);
  return o;
}

template <int MODE, bool PAIR>
struct Smem {
  using C = Cfg<MODE, PAIR>;
  uint32_t base;
  __device__ uint32_t a(int s) const { return base + C::OFF_A + s * C::A_STAGE; }
  __device__ uint32_t b(int s) const { return base + C::OFF_B + s * C::B_STAGE; }
  __device__ uint32_t stage(int w, int i) const {
    return base + C::OFF_STAGE + (w * 2 + i) * C::STAGE_BUF;
  }
  __device__ uint32_t bar(int i) const { return base + C::OFF_BAR + 8 * i; }
  __device__ uint32_t a_full(int s) const { return bar(s); }
  __device__ uint32_t a_empty(int s) const { return bar(C::A_STAGES + s); }
  __device__ uint32_t b_full(int s) const { return bar(2 * C::A_STAGES + s); }
  __device__ uint32_t b_empty(int s) const { return bar(2 * C::A_STAGES + C::B_STAGES + s); }
  __device__ uint32_t acc_full(int b) const {
    return bar(2 * C::A_STAGES + 2 * C::B_STAGES + b);
  }
  __device__ uint32_t acc_empty(int b) const {
    return bar(2 * C::A_STAGES + 2 * C::B_STAGES + C::NACC + b);
  }
  __device__ uint32_t code(int s) const { return base + C::OFF_CODE + s * C::CODE_STAGE; }
  __device__ uint32_t c_full(int s) const {
    return bar(2 * C::A_STAGES + 2 * C::B_STAGES + 2 * C::NACC + s);
  }
  __device__ uint32_t c_empty(int s) const {
    return bar(2 * C::A_STAGES + 2 * C::B_STAGES + 2 * C::NACC + C::CST + s);
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

// silu(z) = z sigmoid(z) = z/2 (1 + tanh(z/2)): one special-function
// instruction per value (the hardware tanh approximation, relative error
// about 2^-11, the rounding of the fp16 result) instead of an exponential
// and a reciprocal -- the gate/up epilogue, which the MMAs wait for, was
// bound by that unit.
__device__ __forceinline__ float silu_tanh(float z) {
  const float hz = 0.5f * z;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hz));
  return fmaf(hz, t, hz);
}

// TMA load of B: a 2-D tile (16 rows) into this CTA's shared memory, its
// bytes counted on this CTA's barrier at `bar`.
__device__ __forceinline__ void tma_tile_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// TMA load of this CTA's half of a pair's B tile (a 16-row slab into its own
// shared memory); the bytes are counted on the barrier at `bar_cluster`, a
// shared::cluster address in either CTA of the pair (the MMA-issuing one).
__device__ __forceinline__ void tma_tile_2d_pair(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
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

// CL: CTAs per cluster, 1 without pairs.
// PAIR (CL = 2, grouped modes): the two CTAs form a tcgen05 pair working on
// the same token tile.  The even CTA issues MMAs of M = 256 over both CTAs'
// A tiles (its own weight unit m and the odd CTA's m + 1, each dequantised
// into its own TMEM); each CTA loads half of the token tile into its own
// shared memory, so that every B byte is written to and read from one SM's
// shared memory only once for 256 weight rows.  The odd CTA's dequantising
// and epilogue warps arrive on the even CTA's barriers; the even CTA's
// commits arrive on both CTAs'.
template <int MODE, int CL, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) grouped_mma_kernel(const __grid_constant__ MmaParams p) {
  static_assert(PAIR ? (CL == 2 && MODE != MMA_ROUTER) : CL == 1,
                "pairs: two CTAs, grouped modes; otherwise one CTA");
  using C = Cfg<MODE, PAIR>;
  constexpr int kPad = PAIR ? 32 : 16;
  // gate/up: the epilogue warps, idle while a unit's MMAs run (its single
  // accumulator pair is drained only at the unit's end), dequantise every
  // other K block, halving the dequantisation latency the MMAs see
  constexpr bool kDeqSplit = (MODE == MMA_GATEUP);
  static_assert(!kDeqSplit || Cfg<MODE, PAIR>::A_STAGES >= 2, "two dequantising groups");
  constexpr int kBStages = C::B_STAGES;
  constexpr int kAStages = C::A_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem<MODE, PAIR> S{smem_u32(smem)};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nunits =
      (MODE == MMA_ROUTER) ? p.nunits_host : (*p.ntiles_dev) * p.units_per_tile;
  // work: the i-th cluster unit of cluster cid is cunit(i) over the tile list
  // (sorted by size: full tiles first, then remainders largest first); the
  // CTA of rank r takes unit cu * CL + r (same tile for the whole cluster,
  // weight unit m = consecutive)
  const int ncu = nunits / CL;
  const int cid = (CL == 1) ? (int)blockIdx.x : (int)cluster_id();
  const int ncl = (CL == 1) ? (int)gridDim.x : (int)cluster_count();
  const int crank = (CL == 1) ? 0 : (int)cluster_rank();
  if (cid >= ncu) return;  // uniform over the cluster
  // With ncu = q ncl + r units, r clusters must take q + 1 of them: those
  // clusters take the r (q + 1) smallest units (the end of the sorted list)
  // and the other ncl - r clusters q of the largest.  A unit's cost is mostly
  // fixed (its K loop of weight blocks) and only partly proportional to its
  // tokens, so dealing the extra units at random made the clusters holding
  // one more unit the kernel's tail.  Within each group, snake order.
  // (Heavy clusters are the first r, so that with fewer units than clusters
  // the ones left without work are the last, as the early return assumes.)
  const int q = ncu / ncl, r = ncu % ncl;
  const int nlight = ncl - r;  // clusters with q units
  const bool heavy = cid < r;
  const int gsize = heavy ? r : nlight, gid = heavy ? cid : cid - r;
  const int gbase = heavy ? nlight * q : 0;
  auto cunit = [&](int i) {
    const int base = gbase + i * gsize;
    return (i & 1) ? base + (gsize - 1 - gid) : base + gid;
  };
  const int nmy = heavy ? q + 1 : q;  // this cluster's units
  const bool leader = !PAIR || crank == 0;  // issues the MMAs

  // some token of the call has an activation scale s != 1 (gate/up epilogue)
  const bool xscaled = (MODE == MMA_GATEUP) && p.xscaled && *p.xscaled != 0;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(S.a_full(s), MODE == MMA_ROUTER ? 1 : (PAIR ? 2 : 1) * kDeqWarps);
      mbar_init(S.a_empty(s), C::NISS);
    }
    for (int s = 0; s < kBStages; ++s) {
      // gate/up: one arrival per CTA of the pair (gathered rows, no byte count)
      mbar_init(S.b_full(s), (MODE == MMA_GATEUP && PAIR) ? 2 : 1);
      mbar_init(S.b_empty(s), C::NISS);
    }
    for (int b = 0; b < C::NACC; ++b) {
      mbar_init(S.acc_full(b), C::NISS);
      mbar_init(S.acc_empty(b), (PAIR ? 2 : 1) * kEpiWarps);
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
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // the peer's barriers are initialised before it arrives
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kbu = p.kb_per_unit;
  const int kbs = kbu / C::KPS;  // pipeline stages per unit

  // Dequantise stage g (the g-th of this CTA's sequence: KPS K blocks) into
  // its A stage in TMEM: thread t (0..255 of a group of 8 warps) takes row t
  // of the unit (two tiles: tile t >> 7) or row t & 127, K half t >> 7 (one
  // tile).  The warp's TMEM lane quarter (lanes 32 (warp % 4) ..) holds rows
  // (t & 127).  Returns false on a timeout.
  auto dequant_kb = [&](int g, int t) -> bool {
    const int row = (C::NA == 2) ? t : (t & 127);
    const int kh = (C::NA == 2) ? 0 : (t >> 7);
    const uint32_t a_lane = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t a_off = (C::NA == 2) ? (uint32_t)((t >> 7) * 32) : (uint32_t)(kh * 16);
    constexpr int kCst = C::CST > 0 ? C::CST : 1;
    constexpr int NW = (C::NA == 2) ? 8 : 4;  // code words of the row (8 values each)
    const int sc = g % kCst, sa = g % kAStages;
    // The codes are loaded and dequantised into registers first, while the
    // MMAs that still read A stage sa run: only the TMEM store waits for the
    // stage, so the chain from those MMAs' commit to the next arrival on
    // a_full is the store alone.
    if (!warp_wait(S.c_full(sc), (g / kCst) & 1, abort_flag, p.err)) return false;
    uint32_t v[C::KPS][4 * NW];  // column 4 i + j = K pair (8 i + 2 j, 8 i + 2 j + 1)
#pragma unroll
    for (int k2 = 0; k2 < C::KPS; ++k2) {
      // row `row` of K block k2 of the ring stage: codes, then the s,b word
      const uint32_t cs = S.code(sc) + k2 * C::CODE_KB;
      const uint4 a0 = ld_shared_v4(cs + row * 32 + kh * 16);
      const uint4 a1 = (C::NA == 2) ? ld_shared_v4(cs + row * 32 + 16) : a0;
      const uint32_t sb = ld_shared_u32(cs + 32 * 128 * C::NA + row * 4);
      const uint32_t s2 = __byte_perm(sb, 0, 0x1010);
      const uint32_t b2 = __byte_perm(sb, 0, 0x3232);
      const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int i = 0; i < NW; ++i) {
        const uint4 d4 = dequant_word(w[i], s2, b2);
        v[k2][4 * i] = d4.x;
        v[k2][4 * i + 1] = d4.y;
        v[k2][4 * i + 2] = d4.z;
        v[k2][4 * i + 3] = d4.w;
      }
    }
    // the code stage is read (the loads above have returned their values)
    __syncwarp();
    if (lane == 0) mbar_arrive(S.c_empty(sc));
    // A stage sa is free once the MMAs of K block g - A_STAGES have completed.
    // Pairs: those MMAs' commit arrives only on the B slot's barrier; the B
    // ring is deeper than the A ring and K block g + B_STAGES - A_STAGES
    // cannot complete before this one is dequantised, so the slot's phase
    // for g - A_STAGES is still the one the parity names.
    if constexpr (PAIR) {
      static_assert(C::B_STAGES > C::A_STAGES, "B ring deeper than the A ring");
      const int gp = g - kAStages;
      if (gp >= 0 && !warp_wait(S.b_empty(gp % C::B_STAGES), (gp / C::B_STAGES) & 1, abort_flag,
                                p.err))
        return false;
    } else {
      if (!warp_wait(S.a_empty(sa), ((g / kAStages) & 1) ^ 1, abort_flag, p.err)) return false;
    }
    // the MMAs that read this A stage before have completed
    tc_fence_after();
#pragma unroll
    for (int k2 = 0; k2 < C::KPS; ++k2) {
      // K block k2's columns follow block k2 - 1's (NA x 32 per block)
      const uint32_t ta =
          tmem + a_lane + C::A_COL0 + sa * C::A_COLS + k2 * (C::NA * 32) + a_off;
      if constexpr (NW == 8)
        tmem_st32(ta, v[k2]);
      else
        tmem_st16(ta, v[k2]);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (leader)
        mbar_arrive(S.a_full(sa));
      else
        mbar_arrive_cluster(mapa_shared(S.a_full(sa), 0));
    }
    return true;
  };

  if (warp == 0 && MODE == MMA_GATEUP) {
    // ------------------------------------------------ B gathered (gate/up)
    // Row n of the token tile is token perm[row0 + n]; this CTA loads rows
    // [crank * npad / 2, ...) of a pair's tile (all of it without a pair)
    // from the fp16 activations by 16-byte cp.async into the 128-byte
    // swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8)); rows
    // past the tile's tokens are zero.  A stage is announced kLag stages after
    // its copies were issued: cp.async.wait_group, the proxy fence that makes
    // the writes visible to the tensor core, then one arrival (in a pair on
    // the even CTA's barrier, which counts one arrival per CTA).  (TMA 4-row
    // gathers, which would count bytes on the even CTA's barrier directly,
    // measured 26 % slower for this kernel: the gather rate bounds them.)
    constexpr int kLag = kBStages > 4 ? 4 : kBStages - 1;  // below the ring depth
    constexpr int kRowsPerLane = ((PAIR ? C::NMAX / 2 : C::NMAX) + 31) / 32;
    const uint32_t fb0 = mapa_shared(S.b_full(0), 0);  // b_full(s) = fb0 + 8 s
    auto announce = [&](uint32_t g) {
      const int s = (int)(g % kBStages);
      if (!PAIR || leader)
        mbar_arrive(S.b_full(s));
      else
        mbar_arrive_cluster(fb0 + 8 * s);
    };
    uint32_t gb = 0;
    bool ok = true;
    for (int i = 0; i < nmy && ok; ++i) {
      const Unit t = get_unit(p, MODE, cunit(i) * CL + crank, kPad);
      const int hn = PAIR ? (t.npad >> 1) : t.npad;
      const int hr0 = t.row0 + (PAIR ? crank * hn : 0);
      int tok[kRowsPerLane];
#pragma unroll
      for (int m = 0; m < kRowsPerLane; ++m) {
        const int r = lane + 32 * m;
        tok[m] = (r < hn && hr0 + r < t.row0 + t.nrows) ? p.perm[hr0 + r] : -1;
      }
      for (int kb = 0; kb < kbu; ++kb) {
        const int s = gb % kBStages;
        if (!warp_wait(S.b_empty(s), ((gb / kBStages) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t bs = S.b(s);
#pragma unroll
        for (int m = 0; m < kRowsPerLane; ++m) {
          const int r = lane + 32 * m;
          if (r < hn) {
            const uint16_t* src = p.xg + (long long)(tok[m] < 0 ? 0 : tok[m]) * p.ldx + kb * 64;
            const uint32_t nb = tok[m] < 0 ? 0u : 16u;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              cp_async16(bs + r * 128 + ((c ^ (r & 7)) << 4), src + c * 8, nb);
          }
        }
        cp_async_commit();
        ++gb;
        if (gb > (uint32_t)kLag) {
          cp_async_wait<kLag>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) announce(gb - 1 - kLag);
        }
      }
    }
    // the last stages (after a timeout every issued copy still completes)
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && ok)
      for (uint32_t g = gb > (uint32_t)kLag ? gb - kLag : 0; g < gb; ++g) announce(g);
  } else if (warp == 0) {
    // ------------------------------------------------------ B (+ router A)
    uint32_t gb = 0, ga = 0;
    bool ok = true;
    Unit tn = get_unit(p, MODE, cunit(0) * CL + crank, kPad);
    for (int i = 0; i < nmy && ok; ++i) {
      const Unit t = tn;
      if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank, kPad);
      const int k0 = t.ks * kbu;
      const uint8_t* asrc = p.wA + (long long)t.m * p.a_unit_stride + (long long)k0 * p.a_chunk;
      for (int kb = 0; kb < kbs; ++kb) {
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
        if constexpr (PAIR) {
          // this CTA's half of the tile (rows crank * npad / 2 ..), counted on
          // the even CTA's barrier, which expects the bytes of both halves
          if (lane == 0 && leader)
            mbar_arrive_expect_tx(S.b_full(s), (uint32_t)t.npad * 128 * C::KPS);
          __syncwarp();
          const int half = t.npad >> 1;
          const uint32_t fb = mapa_shared(S.b_full(s), 0);
#pragma unroll
          for (int k2 = 0; k2 < C::KPS; ++k2)
            for (int sl = lane; sl < (half >> 4); sl += 32)
              tma_tile_2d_pair(bs + k2 * C::B_SUB + sl * 2048, &p.tmB,
                               (k0 + kb * C::KPS + k2) * 64, t.row0 + crank * half + 16 * sl, fb);
        } else {
          // the whole tile, one 2-D tile per 16-row slab
          if (lane == 0) mbar_arrive_expect_tx(S.b_full(s), (uint32_t)t.npad * 128 * C::KPS);
          __syncwarp();
          const int nslab = t.npad >> 4;
#pragma unroll
          for (int k2 = 0; k2 < C::KPS; ++k2)
            for (int sl = lane; sl < nslab; sl += 32)
              tma_tile_2d(bs + k2 * C::B_SUB + sl * 2048, &p.tmB,
                              (k0 + kb * C::KPS + k2) * 64, t.row0 + 16 * sl, S.b_full(s));
        }
        ++gb;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (every wait and operand warp-uniform) and
    // one elected lane issues each MMA and commit: issuing from one divergent
    // lane cost ~100-150 cycles per MMA (per-K-block clock64 stamps).
    if (leader) {
      uint32_t sa = 0, pa = 0, sb = 0, pb = 0;  // ring slots and phase parities
      Unit tn = get_unit(p, MODE, cunit(0) * CL + crank, kPad);
      for (int i = 0; i < nmy; ++i) {
        const Unit t = tn;  // the next unit's descriptor loads during this one
        if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank, kPad);
        const int ab = (C::NACC == 2) ? (int)(i & 1) : 0;
        const uint32_t aph = ((C::NACC == 2) ? (i >> 1) : i) & 1;
        if (!warp_wait(S.acc_empty(ab), aph ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(PAIR ? 256 : 128, t.npad, MODE == MMA_ROUTER ? 1 : 0);
        bool ok = true;
        for (int kb = 0; kb < kbs; ++kb) {
          // both operands' barriers tested at once (the two tests' latencies
          // overlap), the outcome taken for the whole warp
          const bool ra = mbar_try_wait(S.a_full(sa), pa);
          const bool rb = mbar_try_wait(S.b_full(sb), pb);
          if (!__all_sync(0xffffffffu, ra && rb) &&
              (!warp_wait(S.a_full(sa), pa, abort_flag, p.err) ||
               !warp_wait(S.b_full(sb), pb, abort_flag, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k2 = 0; k2 < C::KPS; ++k2) {
            // K step kk: both operands advance by 32 bytes (2 in the
            // descriptor's address field, which holds the address / 16)
            const uint64_t bd = sdesc_k_sw128(S.b(sb) + k2 * C::B_SUB);
            const uint32_t acc = (kb | k2) ? 1u : 0u;
#pragma unroll
            for (int j = 0; j < C::NA; ++j) {
              // NA == 2: tile j -> columns NMAX j; NACC == 2: buffer ab -> columns NMAX ab
              const uint32_t dcol = tmem + C::NMAX * (C::NA == 2 ? j : ab);
              if constexpr (C::TMEM_A) {
                // A: 8 TMEM columns per K step of 16; K block k2 after k2 - 1
                const uint32_t at = tmem + C::A_COL0 + sa * C::A_COLS + k2 * (C::NA * 32) + j * 32;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  if constexpr (PAIR)
                    tc_mma_f16_ts_pair_w(dcol, at + 8 * kk, bd + 2 * kk, idesc, (acc | kk) ? 1u : 0u);
                  else
                    tc_mma_f16_ts_w(dcol, at + 8 * kk, bd + 2 * kk, idesc, (acc | kk) ? 1u : 0u);
                }
              } else {
                const uint64_t ad = sdesc_k_sw128(S.a(sa) + j * 16384);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_f16_w(dcol, ad + 2 * kk, bd + 2 * kk, idesc, (acc | kk) ? 1u : 0u);
              }
            }
          }
          if constexpr (PAIR) {
            // one commit frees both stages: the dequantising warps wait on
            // the B slot's barrier (see dequant_kb)
            tc_commit_pair_mc_w(S.b_empty(sb), 3);
          } else {
            tc_commit_w(S.a_empty(sa));
            tc_commit_w(S.b_empty(sb));
          }
          if (++sa == kAStages) { sa = 0; pa ^= 1; }
          if (++sb == (uint32_t)kBStages) { sb = 0; pb ^= 1; }
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair_mc_w(S.acc_full(ab), 3);
        else
          tc_commit_w(S.acc_full(ab));
      }
      // every issued MMA has finished before TMEM is released (in both CTAs
      // of a pair)
      if constexpr (PAIR)
        tc_commit_pair_mc_w(S.drain(), 3);
      else
        tc_commit_w(S.drain());
    }
    if (lane == 0) mbar_wait_bounded(S.drain(), 0, abort_flag, kWaitLimitNs);
  } else if (warp == 2 && MODE != MMA_ROUTER) {
    // ------------------------------------------------ code ring
    if (lane == 0) {
      const int total = nmy * kbs;
      for (int g = 0; g < total; ++g) {
        constexpr int kCst = C::CST > 0 ? C::CST : 1;
        const int s = g % kCst;
        if (!thread_wait(S.c_empty(s), ((g / kCst) & 1) ^ 1, abort_flag, p.err)) break;
        const int j = g / kbs;
        const Unit u = get_unit(p, MODE, cunit(j) * CL + crank, kPad);
        mbar_arrive_expect_tx(S.c_full(s), C::CODE_STAGE);
#pragma unroll
        for (int k2 = 0; k2 < C::KPS; ++k2) {
          const int kbk = (g - j * kbs) * C::KPS + k2;  // K block within the unit
          const uint32_t dst = S.code(s) + k2 * C::CODE_KB;
          if (C::NA == 2) {  // the whole chunk of unit m
            const uint8_t* ch = p.wA + (long long)u.expert * p.a_expert_stride +
                                (long long)u.m * p.a_unit_stride + (long long)kbk * p.a_chunk;
            bulk_g2s(dst, ch, kCodeChunk, S.c_full(s));
          } else {  // rows 128 (m % 2) .. +127 of chunk unit m / 2: codes, s,b words
            const uint8_t* ch = p.wA + (long long)u.expert * p.a_expert_stride +
                                (long long)(u.m >> 1) * p.a_unit_stride +
                                (long long)kbk * p.a_chunk;
            const int h = u.m & 1;
            bulk_g2s(dst, ch + h * 4096, 4096, S.c_full(s));
            bulk_g2s(dst + 4096, ch + 8192 + h * 512, 512, S.c_full(s));
          }
        }
      }
    }
  } else if (warp >= 4 && warp < 4 + kDeqWarps) {
    // ------------------------------------------------ dequantise
    if constexpr (MODE != MMA_ROUTER) {
      const int total = nmy * kbs;
      // gate/up: these warps take the even K blocks, the epilogue warps the
      // odd ones (kbs is even, so the parity of g is that of the K block)
      for (int g = 0; g < total; g += kDeqSplit ? 2 : 1)
        if (!dequant_kb(g, threadIdx.x - 32 * 4)) break;
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------- epilogue
    const int e = warp - kEpiWarp0;    // 0..7
    const int q = warp & 3;            // TMEM lane quarter
    const int half = e >> 2;           // columns [128*half, 128*half + 128)
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t nst = 0;
    Unit tn = get_unit(p, MODE, cunit(0) * CL + crank, kPad);
    for (int i = 0; i < nmy; ++i) {
      const Unit t = tn;
      if (i + 1 < nmy) tn = get_unit(p, MODE, cunit(i + 1) * CL + crank, kPad);
      if constexpr (kDeqSplit) {
        // the odd K blocks of this unit (the MMAs of the next unit cannot
        // start before this unit's epilogue has drained its accumulators)
        bool ok = true;
        for (int kb = 1; kb < kbs && ok; kb += 2)
          ok = dequant_kb(i * kbs + kb, threadIdx.x - 32 * kEpiWarp0);
        if (!ok) break;
      }
      const int c0 = half * C::EPI_COLS;
      const int c1 = min(c0 + C::EPI_COLS, t.npad);
      // row data of the warp's 128 columns, fetched while the MMAs run:
      // lane l holds rows c0 + l + 32 v, v = 0..3
      // (down: the routing weight and contribution row; gate/up, when some
      // token of the call was scaled: the power of two that scaled the row's
      // fp16 activations)
      constexpr float kR0 = (MODE == MMA_GATEUP) ? 1.f : 0.f;
      float rsc4[4] = {kR0, kR0, kR0, kR0};
      int rdst4[4] = {0, 0, 0, 0};
      if (MODE == MMA_DOWN || (MODE == MMA_GATEUP && xscaled)) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int n = c0 + lane + 32 * v;
          if (n < t.nrows) {
            if (MODE == MMA_DOWN) {
              rsc4[v] = p.row_scale[t.row0 + n];
              rdst4[v] = p.dst_row[t.row0 + n];
            } else {
              rsc4[v] = p.row_xscale[t.row0 + n];
            }
          }
        }
      }
      const int ab = (C::NACC == 2) ? (int)(i & 1) : 0;
      const uint32_t aph = ((C::NACC == 2) ? (i >> 1) : i) & 1;
      if (!warp_wait(S.acc_full(ab), aph, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + C::NMAX * ab;
      // SC: some token of the call was scaled (gate/up; a separate copy of the
      // chunk loop, so that the usual case runs without the scaling)
      auto chunks = [&](auto sc_tag) {
        constexpr bool SC = decltype(sc_tag)::value;
        for (int n0 = c0; n0 < c1; n0 += 16) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tacc + n0, r0);
          if (C::NA == 2) tmem_ld16(tacc + C::NMAX + n0, r1);
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
                float h;
                if constexpr (SC) {
                  // The row's activations entered as x / s (s a power of two),
                  // so the accumulators are v0 = g / s and v1 = u / s.  H holds
                  // silu(g) u / s^2 = silu(s v0) * (v1 / s), bounded by |v0 v1|
                  // (|silu(z)| <= |z|); the down projection's row weight carries
                  // the s^2 back.
                  const float ps = __shfl_sync(0xffffffffu, rsc, j);
                  const float pinv = __int_as_float(0x7F000000 - __float_as_int(ps));  // 1/s, exact
                  h = silu_tanh(v0 * ps) * (v1 * pinv);
                } else {
                  h = silu_tanh(v0) * v1;
                }
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
      };
      if (MODE == MMA_GATEUP && xscaled)
        chunks(std::true_type{});
      else
        chunks(std::false_type{});
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(S.acc_empty(ab));
        else
          mbar_arrive_cluster(mapa_shared(S.acc_empty(ab), 0));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // no CTA leaves while peers may still write to it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
}

template <int MODE, int CL, bool PAIR>
cudaError_t launch_mode(const MmaParams& p, int grid, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_mma_kernel<MODE, CL, PAIR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MODE, PAIR>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // no more clusters than can be resident at once (persistent CTAs)
  static int max_grid = -1;
  if (max_grid < 0) {
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(CL);
    q.blockDim = dim3(kThreads);
    q.dynamicSmemBytes = Cfg<MODE, PAIR>::SMEM;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = CL;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    q.attrs = a;
    q.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, grouped_mma_kernel<MODE, CL, PAIR>, &q) != cudaSuccess ||
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
  cfg.dynamicSmemBytes = Cfg<MODE, PAIR>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_mma_kernel<MODE, CL, PAIR>, p);
}

// CTA pairs (tcgen05 cta_group::2) for the grouped GEMMs unless
// MOE_GEMM_2SM=0; they need an even number of weight units per tile.
bool pairs_for(int units_per_tile) {
  static int env = -1;
  if (env < 0) {
    const char* e = getenv("MOE_GEMM_2SM");
    env = (e && atoi(e) == 0) ? 0 : 1;
  }
  return env == 1 && units_per_tile % 2 == 0;
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
  if (mode == MMA_ROUTER) return launch_mode<MMA_ROUTER, 1, false>(p, grid, st);
  if (pairs_for(p.units_per_tile)) {
    if (mode == MMA_GATEUP) return launch_mode<MMA_GATEUP, 2, true>(p, grid, st);
    return launch_mode<MMA_DOWN, 2, true>(p, grid, st);
  }
  if (mode == MMA_GATEUP) return launch_mode<MMA_GATEUP, 1, false>(p, grid, st);
  return launch_mode<MMA_DOWN, 1, false>(p, grid, st);
}

}  // namespace moe
