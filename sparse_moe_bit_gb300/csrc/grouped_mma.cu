// Grouped tensor-core GEMM for sm_103a: tcgen05.mma with TMEM accumulators,
// operands staged in shared memory by bulk (TMA) copies and cp.async, 4-bit
// weights dequantised tile by tile inside the pipeline.
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
// Warp roles (448 threads, one CTA per SM, persistent over the unit list):
//   warp 0      lane 0: bulk copies of A (codes+scales, or router rows)
//   warp 1      lane 0: tcgen05.mma issue; the warp owns the TMEM allocation
//   warps 2..5  dequantise codes -> fp16 A tiles (128-byte swizzled, K-major)
//   warps 6..9  gather B rows with cp.async into 128-byte swizzled tiles
//   warps 10..13 epilogue: tcgen05.ld, activation / scaling, global stores
// Pipelines: kStages stages of {codes, A, B}; TMEM holds two fp32
// accumulators of 256 columns (A0 at column 0, A1 at column 256).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 448;
constexpr int kAStage = 32768;  // two 128 x 64 x 16-bit tiles
constexpr int kBStage = 32768;  // up to 256 x 64 x 16-bit
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffCodes = kOffB + kStages * kBStage;
constexpr int kOffBar = kOffCodes + kStages * kCodeChunk;
constexpr int kNumBars = 5 * kStages + 3;
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
  __device__ uint32_t bar(int i) const { return base + kOffBar + 8 * i; }
  __device__ uint32_t code_full(int s) const { return bar(s); }
  __device__ uint32_t code_empty(int s) const { return bar(kStages + s); }
  __device__ uint32_t a_full(int s) const { return bar(2 * kStages + s); }
  __device__ uint32_t b_full(int s) const { return bar(3 * kStages + s); }
  __device__ uint32_t ab_empty(int s) const { return bar(4 * kStages + s); }
  __device__ uint32_t acc_full() const { return bar(5 * kStages); }
  __device__ uint32_t acc_empty() const { return bar(5 * kStages + 1); }
  __device__ uint32_t drain() const { return bar(5 * kStages + 2); }
};

__device__ __forceinline__ void record_timeout(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  atomicOr(err, MOE_DEVERR_WAIT_TIMEOUT);
}

// All 32 lanes wait for the phase; the give-up decision is taken by lane 0 and
// shared, so the warp leaves together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((i & 63u) == 63u) {
      int bail = 0;
      if (lane == 0) {
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        else if (now - t0 > kWaitLimitNs) bail = 1;
        if (*abort_flag) bail = 1;
      }
      bail = __shfl_sync(0xffffffffu, bail, 0);
      if (bail) {
        if (lane == 0) record_timeout(abort_flag, err);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            int* err) {
  if (mbar_wait_bounded(bar, parity, abort_flag, kWaitLimitNs)) return true;
  record_timeout(abort_flag, err);
  return false;
}

// fp16 pair (1024 + q_lo, 1024 + q_hi) from the nibbles at bit 4j and 16+4j.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t v, int j, uint32_t s2, uint32_t b2) {
  const uint32_t t = ((v >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
  __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&t),
                      __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  __half2 r = __hfma2(q, *reinterpret_cast<const __half2*>(&s2),
                      *reinterpret_cast<const __half2*>(&b2));
  return *reinterpret_cast<uint32_t*>(&r);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_mma_kernel(const MmaParams p) {
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(S.code_full(s), 1);
      mbar_init(S.code_empty(s), 4);
      mbar_init(S.a_full(s), MODE == MMA_ROUTER ? 1 : 4);
      mbar_init(S.b_full(s), 4);
      mbar_init(S.ab_empty(s), 1);
    }
    mbar_init(S.acc_full(), 1);
    mbar_init(S.acc_empty(), 4);
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
    // ---------------------------------------------------------- A producer
    if (lane == 0) {
      uint32_t g = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const Unit t = get_unit(p, MODE, u);
        const uint8_t* src = p.wA + (long long)t.expert * p.a_expert_stride +
                             (long long)t.m * p.a_unit_stride +
                             (long long)t.ks * kbu * p.a_chunk;
        for (int kb = 0; kb < kbu; ++kb, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (MODE == MMA_ROUTER) {
            if (!thread_wait(S.ab_empty(s), ph ^ 1, abort_flag, p.err)) goto a_done;
            mbar_arrive_expect_tx(S.a_full(s), kRouterChunk);
            bulk_g2s(S.a(s), src + (long long)kb * p.a_chunk, kRouterChunk, S.a_full(s));
          } else {
            if (!thread_wait(S.code_empty(s), ph ^ 1, abort_flag, p.err)) goto a_done;
            mbar_arrive_expect_tx(S.code_full(s), kCodeChunk);
            bulk_g2s(S.codes(s), src + (long long)kb * p.a_chunk, kCodeChunk, S.code_full(s));
          }
        }
      }
    a_done:;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t g = 0, i = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
        const Unit t = get_unit(p, MODE, u);
        if (!thread_wait(S.acc_empty(), (i & 1) ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(128, t.npad, MODE == MMA_ROUTER ? 1 : 0);
        bool ok = true;
        for (int kb = 0; kb < kbu; ++kb, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!thread_wait(S.a_full(s), ph, abort_flag, p.err) ||
              !thread_wait(S.b_full(s), ph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a0 = sdesc_k_sw128(S.a(s) + kk * 32);
            const uint64_t a1 = sdesc_k_sw128(S.a(s) + 16384 + kk * 32);
            const uint64_t bd = sdesc_k_sw128(S.b(s) + kk * 32);
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            tc_mma_f16(tmem, a0, bd, idesc, acc);
            tc_mma_f16(tmem + 256, a1, bd, idesc, acc);
          }
          tc_commit(S.ab_empty(s));
        }
        if (!ok) break;
        tc_commit(S.acc_full());
      }
      // every issued MMA has finished before TMEM is released
      tc_commit(S.drain());
      mbar_wait_bounded(S.drain(), 0, abort_flag, kWaitLimitNs);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- dequantise
    if (MODE != MMA_ROUTER) {
      const int dw = warp - 2;
      uint32_t g = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        for (int kb = 0; kb < kbu; ++kb, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!warp_wait(S.code_full(s), ph, abort_flag, p.err)) goto dq_done;
          if (!warp_wait(S.ab_empty(s), ph ^ 1, abort_flag, p.err)) goto dq_done;
          const uint32_t codes = S.codes(s);
          const uint32_t a = S.a(s);
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
            mbar_arrive(S.a_full(s));
            mbar_arrive(S.code_empty(s));
          }
        }
      }
    dq_done:;
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------- B loader
    const int bt = threadIdx.x - 192;
    uint32_t g = 0;
    int prev_s = -1;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit t = get_unit(p, MODE, u);
      const long long k0 = (long long)t.ks * kbu * 64;
      for (int kb = 0; kb < kbu; ++kb, ++g) {
        const int s = g % kStages;
        const uint32_t ph = (g / kStages) & 1;
        if (!warp_wait(S.ab_empty(s), ph ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t bs = S.b(s);
        for (int i = bt; i < t.npad * 8; i += 128) {
          const int n = i >> 3;
          const int c = i & 7;
          const bool valid = n < t.nrows;
          const uint16_t* src = p.B;
          if (valid) {
            const int grow = t.row0 + n;
            const long long srow = p.b_rowmap ? (long long)p.b_rowmap[grow] : (long long)grow;
            src = p.B + srow * p.ldb + k0 + kb * 64 + c * 8;
          }
          cp_async16(bs + n * 128 + ((c ^ (n & 7)) << 4), src, valid ? 16u : 0u);
        }
        cp_async_commit();
        if (prev_s >= 0) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(S.b_full(prev_s));
        }
        prev_s = s;
      }
    }
    cp_async_wait<0>();
    if (ok && prev_s >= 0) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(S.b_full(prev_s));
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t i = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
      const Unit t = get_unit(p, MODE, u);
      if (!warp_wait(S.acc_full(), i & 1, abort_flag, p.err)) break;
      tc_fence_after();
      for (int n0 = 0; n0 < t.npad; n0 += 16) {
        uint32_t r0[16], r1[16];
        tmem_ld16(tmem + lane_base + n0, r0);
        tmem_ld16(tmem + lane_base + 256 + n0, r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = n0 + j;
          if (n < t.nrows) {
            const float v0 = __uint_as_float(r0[j]);
            const float v1 = __uint_as_float(r1[j]);
            const int row = t.row0 + n;
            if (MODE == MMA_GATEUP) {
              const float h = v0 / (1.0f + __expf(-v0)) * v1;
              const int f = t.m * 128 + q * 32 + lane;
              p.H[(long long)row * p.ldh + f] = __half_as_ushort(__float2half_rn(h));
            } else if (MODE == MMA_DOWN) {
              const float sc = p.row_scale[row];
              const long long drow = p.dst_row[row];
              const int f = t.m * 256 + q * 32 + lane;
              uint16_t* yr = p.Y + drow * p.ldy;
              yr[f] = __bfloat16_as_ushort(__float2bfloat16_rn(sc * v0));
              yr[f + 128] = __bfloat16_as_ushort(__float2bfloat16_rn(sc * v1));
            } else {
              const int e = t.m * 256 + q * 32 + lane;
              float* o = p.out_f32 + ((long long)t.ks * p.rows_total + row) * p.E;
              if (e < p.E) o[e] = v0;
              if (e + 128 < p.E) o[e + 128] = v1;
            }
          }
        }
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

}  // namespace

cudaError_t launch_grouped_mma(int mode, const MmaParams& p, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  switch (mode) {
    case MMA_ROUTER: return launch_mode<MMA_ROUTER>(p, grid, st);
    case MMA_GATEUP: return launch_mode<MMA_GATEUP>(p, grid, st);
    default: return launch_mode<MMA_DOWN>(p, grid, st);
  }
}

}  // namespace moe
