// Grouped tensor-core GEMM for sm_103a: tcgen05.mma with TMEM accumulators,
// operands staged in shared memory by the tensor memory accelerator (bulk
// copies for the weight codes, 2-D tensor tiles and 4-row gathers for the
// token rows), 4-bit weights dequantised tile by tile inside the pipeline.
//
// One work unit computes two 128-row weight tiles (A0, A1) against one token
// tile of up to 256 rows (B), over K in blocks of 64 (one quantisation group
// per block):
//   router : A = router rows e..e+255 (bf16), B = token rows of x (bf16),
//            out = fp32 partial logits of one K split.
//   gate/up: A0 = gate rows f..f+127, A1 = up rows f..f+127 of one expert
//            (dequantised to fp16), B = the expert's grouped token rows of x
//            (fp16, gathered through the permutation); epilogue
//            H = silu(A0 x) * (A1 x) -> fp16.
//   down   : A0, A1 = down rows f..f+255 (dequantised), B = the expert's rows
//            of H; epilogue Y[dst] = w_row * (A x) -> bf16, written to the
//            token's contribution row (deterministic combine later).
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Dequantize weights during matrix multiplication" (one small weight tile
// at a time is expanded to 16-bit in on-chip memory and multiplied with the
// routed activation rows; fp32 accumulation; the full matrix is never
// written out) and §"Match tile size to expert load" (tile shape from the
// expert's row count: the token dimension N of each tile is the expert's
// remaining row count rounded up to 16, at most 256).
//
// Warp roles (512 threads, one CTA per SM, persistent over the unit list):
//   warp 0      B producer (lane 0 issues TMA; the warp stages row indices)
//               and, for the router, the A bulk copies
//   warp 1      lane 0 issues tcgen05.mma; the warp owns the TMEM allocation
//   warp 2      lane 0 issues the bulk copies of the weight codes
//   warps 4..7  dequantise codes -> fp16 A tiles (128-byte swizzled, K-major)
//   warps 8..15 epilogue: tcgen05.ld, activation / scaling, staging in shared
//               memory, bulk stores of 64-byte row segments
// Rings: A 2 stages, B 3 stages, codes 3 stages.  TMEM: two fp32 accumulators
// of 256 columns (A0 at column 0, A1 at column 256).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kAStages = 2, kBStages = 3, kCStages = 3;
constexpr int kAStage = 32768;  // two 128 x 64 x 16-bit tiles
constexpr int kBStage = 32768;  // up to 256 x 64 x 16-bit
constexpr int kEpiWarps = 8;
constexpr int kStageBuf = 2048;  // per epilogue warp and buffer: 16 rows x 64 x 16-bit
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kAStages * kAStage;
constexpr int kOffCodes = kOffB + kBStages * kBStage;
constexpr int kOffStage = kOffCodes + kCStages * kCodeChunk;
constexpr int kOffRows = kOffStage + kEpiWarps * 2 * kStageBuf;  // 256 gather row indices
constexpr int kOffBar = kOffRows + 256 * 4;
constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kCStages + 3;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

static_assert(kSmemBytes <= 232448, "shared memory budget");

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

struct Smem {
  uint32_t base;
  __device__ uint32_t a(int s) const { return base + kOffA + s * kAStage; }
  __device__ uint32_t b(int s) const { return base + kOffB + s * kBStage; }
  __device__ uint32_t codes(int s) const { return base + kOffCodes + s * kCodeChunk; }
  __device__ uint32_t stage(int w, int i) const {
    return base + kOffStage + (w * 2 + i) * kStageBuf;
  }
  __device__ uint32_t bar(int i) const { return base + kOffBar + 8 * i; }
  __device__ uint32_t a_full(int s) const { return bar(s); }
  __device__ uint32_t a_empty(int s) const { return bar(kAStages + s); }
  __device__ uint32_t b_full(int s) const { return bar(2 * kAStages + s); }
  __device__ uint32_t b_empty(int s) const { return bar(2 * kAStages + kBStages + s); }
  __device__ uint32_t c_full(int s) const { return bar(2 * kAStages + 2 * kBStages + s); }
  __device__ uint32_t c_empty(int s) const {
    return bar(2 * kAStages + 2 * kBStages + kCStages + s);
  }
  __device__ uint32_t acc_full() const { return bar(kNumBars - 3); }
  __device__ uint32_t acc_empty() const { return bar(kNumBars - 2); }
  __device__ uint32_t drain() const { return bar(kNumBars - 1); }
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

// fp16 pair (q_lo, q_hi) * s + beta from the nibbles at bit 4j and 16+4j
__device__ __forceinline__ uint32_t dequant_pair(uint32_t v, int j, uint32_t s2, uint32_t b2) {
  const uint32_t t = ((v >> (4 * j)) & 0x000F000Fu) | 0x64006400u;  // 1024 + q
  __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&t),
                      __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  __half2 r = __hfma2(q, *reinterpret_cast<const __half2*>(&s2),
                      *reinterpret_cast<const __half2*>(&b2));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void tma_tile_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int x, int4 rows,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(rows.x), "r"(rows.y), "r"(rows.z), "r"(rows.w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_mma_kernel(const __grid_constant__ MmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem S{smem_u32(smem)};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nunits =
      (MODE == MMA_ROUTER) ? p.nunits_host : (*p.ntiles_dev) * p.units_per_tile;
  if ((int)blockIdx.x >= nunits) return;  // uniform over the CTA

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* rows_s = reinterpret_cast<int*>(smem + kOffRows);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(S.a_full(s), MODE == MMA_ROUTER ? 1 : 4);
      mbar_init(S.a_empty(s), 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(S.b_full(s), 1);
      mbar_init(S.b_empty(s), 1);
    }
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(S.c_full(s), 1);
      mbar_init(S.c_empty(s), 4);
    }
    mbar_init(S.acc_full(), 1);
    mbar_init(S.acc_empty(), kEpiWarps);
    mbar_init(S.drain(), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kbu = p.kb_per_unit;

  if (warp == 0) {
    // ------------------------------------------------------ B (+ router A)
    uint32_t gb = 0, ga = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit t = get_unit(p, MODE, u);
      if (MODE == MMA_GATEUP) {
        // row indices of the unit's tokens; padding rows repeat a valid row
        __syncwarp();
        for (int i = lane; i < t.npad; i += 32)
          rows_s[i] = p.b_rowmap[t.row0 + (i < t.nrows ? i : 0)];
        __syncwarp();
      }
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
        if (MODE == MMA_GATEUP) {
          // 4-row gathers, issued by 16 lanes (lane i: rows 4i, 4i + 64, ...)
          if (lane == 0) mbar_arrive_expect_tx(S.b_full(s), (uint32_t)t.npad * 128);
          __syncwarp();
          if (lane < 16) {
            for (int n = 4 * lane; n < t.npad; n += 64) {
              const int4 r4 = *reinterpret_cast<const int4*>(rows_s + n);
              tma_gather4(bs + n * 128, &p.tmB, x, r4, S.b_full(s));
            }
          }
        } else if (lane == 0) {
          {
            const int nbox = (t.npad + 31) >> 5;
            mbar_arrive_expect_tx(S.b_full(s), (uint32_t)nbox * 4096);
            for (int i = 0; i < nbox; ++i)
              tma_tile_2d(bs + i * 4096, &p.tmB, x, t.row0 + 32 * i, S.b_full(s));
          }
        }
        ++gb;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t ga = 0, gb = 0, i = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
        const Unit t = get_unit(p, MODE, u);
        if (!thread_wait(S.acc_empty(), (i & 1) ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(128, t.npad, MODE == MMA_ROUTER ? 1 : 0);
        bool ok = true;
        for (int kb = 0; kb < kbu; ++kb, ++ga, ++gb) {
          const int sa = ga % kAStages, sb = gb % kBStages;
          if (!thread_wait(S.a_full(sa), (ga / kAStages) & 1, abort_flag, p.err) ||
              !thread_wait(S.b_full(sb), (gb / kBStages) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a0 = sdesc_k_sw128(S.a(sa) + kk * 32);
            const uint64_t a1 = sdesc_k_sw128(S.a(sa) + 16384 + kk * 32);
            const uint64_t bd = sdesc_k_sw128(S.b(sb) + kk * 32);
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            tc_mma_f16(tmem, a0, bd, idesc, acc);
            tc_mma_f16(tmem + 256, a1, bd, idesc, acc);
          }
          tc_commit(S.a_empty(sa));
          tc_commit(S.b_empty(sb));
        }
        if (!ok) break;
        tc_commit(S.acc_full());
      }
      // every issued MMA has finished before TMEM is released
      tc_commit(S.drain());
      mbar_wait_bounded(S.drain(), 0, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- codes
    if (MODE != MMA_ROUTER && lane == 0) {
      uint32_t gc = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const Unit t = get_unit(p, MODE, u);
        const uint8_t* src = p.wA + (long long)t.expert * p.a_expert_stride +
                             (long long)t.m * p.a_unit_stride;
        for (int kb = 0; kb < kbu; ++kb, ++gc) {
          const int s = gc % kCStages;
          if (!thread_wait(S.c_empty(s), ((gc / kCStages) & 1) ^ 1, abort_flag, p.err)) goto c_done;
          mbar_arrive_expect_tx(S.c_full(s), kCodeChunk);
          bulk_g2s(S.codes(s), src + (long long)kb * p.a_chunk, kCodeChunk, S.c_full(s));
        }
      }
    c_done:;
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- dequantise
    if (MODE != MMA_ROUTER) {
      const int dw = warp - 4;
      uint32_t ga = 0, gc = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        for (int kb = 0; kb < kbu; ++kb, ++ga, ++gc) {
          const int sc = gc % kCStages, sa = ga % kAStages;
          if (!warp_wait(S.c_full(sc), (gc / kCStages) & 1, abort_flag, p.err)) goto dq_done;
          if (!warp_wait(S.a_empty(sa), ((ga / kAStages) & 1) ^ 1, abort_flag, p.err)) goto dq_done;
          const uint32_t codes = S.codes(sc);
          const uint32_t a = S.a(sa);
          const int c = lane & 7;
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int r = 4 * (dw + 4 * it) + (lane >> 3);
            const uint32_t v = ld_shared_u32(codes + r * 32 + c * 4);
            const uint32_t sb = ld_shared_u32(codes + 8192 + r * 4);
            const uint32_t s2 = __byte_perm(sb, 0, 0x1010);
            const uint32_t b2 = __byte_perm(sb, 0, 0x3232);
            const uint32_t w0 = dequant_pair(v, 0, s2, b2);
            const uint32_t w1 = dequant_pair(v, 1, s2, b2);
            const uint32_t w2 = dequant_pair(v, 2, s2, b2);
            const uint32_t w3 = dequant_pair(v, 3, s2, b2);
            const uint32_t dst = a + (r >> 7) * 16384 + (r & 127) * 128 + ((c ^ (r & 7)) << 4);
            st_shared_v4(dst, w0, w1, w2, w3);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(S.a_full(sa));
            mbar_arrive(S.c_empty(sc));
          }
        }
      }
    dq_done:;
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------- epilogue
    const int e = warp - 8;            // 0..7
    const int q = warp & 3;            // TMEM lane quarter
    const int half = e >> 2;           // columns [128*half, 128*half + 128)
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t i = 0, nst = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
      const Unit t = get_unit(p, MODE, u);
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
      if (!warp_wait(S.acc_full(), i & 1, abort_flag, p.err)) break;
      tc_fence_after();
      for (int n0 = c0; n0 < c1; n0 += 16) {
        uint32_t r0[16], r1[16];
        tmem_ld16(tmem + lane_base + n0, r0);
        tmem_ld16(tmem + lane_base + 256 + n0, r1);
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
        // stage [16 rows][32 or 64 values] in shared memory, then 16-byte
        // vector stores of whole 64-byte row segments
        const uint32_t sbuf = S.stage(e, nst & 1);
        __syncwarp();  // the buffer's previous reads are done
        if (nvalid > 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float v0 = __uint_as_float(r0[j]);
            const float v1 = __uint_as_float(r1[j]);
            if (MODE == MMA_GATEUP) {
              const float h = v0 / (1.0f + __expf(-v0)) * v1;
              st_shared_u16(sbuf + j * 64 + lane * 2, __half_as_ushort(__float2half_rn(h)));
            } else {
              const float sc = __shfl_sync(0xffffffffu, rsc, j);
              st_shared_u16(sbuf + j * 128 + lane * 2,
                            __bfloat16_as_ushort(__float2bfloat16_rn(sc * v0)));
              st_shared_u16(sbuf + j * 128 + 64 + lane * 2,
                            __bfloat16_as_ushort(__float2bfloat16_rn(sc * v1)));
            }
          }
        }
        __syncwarp();
        if (MODE == MMA_GATEUP) {
          // 16 rows x 64 bytes: lane -> (row lane/4 + 8i, 16-byte piece lane%4)
#pragma unroll
          for (int it = 0; it < 2; ++it) {
            const int j = (lane >> 2) + 8 * it;
            if (j < nvalid) {
              const uint4 v = ld_shared_v4(sbuf + j * 64 + (lane & 3) * 16);
              const long long row = t.row0 + n0 + j;
              *reinterpret_cast<uint4*>(p.H + row * p.ldh + t.m * 128 + q * 32 + (lane & 3) * 8) = v;
            }
          }
        } else {
          // 16 rows x 2 segments x 64 bytes: lane -> (row lane/8 + 4i, piece lane%8)
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int j = (lane >> 3) + 4 * it;
            const long long dj = __shfl_sync(0xffffffffu, rdst, j);
            if (j < nvalid) {
              const int pc = lane & 7;  // pieces 0..3: first segment, 4..7: second
              const uint4 v = ld_shared_v4(sbuf + j * 128 + pc * 16);
              uint16_t* yr = p.Y + dj * p.ldy + t.m * 256 + q * 32 + (pc >> 2) * 128 + (pc & 3) * 8;
              *reinterpret_cast<uint4*>(yr) = v;
            }
          }
        }
        ++nst;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(S.acc_empty());
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE>
cudaError_t launch_mode(const MmaParams& p, int grid, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_mma_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  grouped_mma_kernel<MODE><<<grid, kThreads, kSmemBytes, st>>>(p);
  return cudaGetLastError();
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
  switch (mode) {
    case MMA_ROUTER: return launch_mode<MMA_ROUTER>(p, grid, st);
    case MMA_GATEUP: return launch_mode<MMA_GATEUP>(p, grid, st);
    default: return launch_mode<MMA_DOWN>(p, grid, st);
  }
}

}  // namespace moe
