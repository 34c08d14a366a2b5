// One-time repacking of the canonical weights (moe_create) into the layouts
// the kernels read.
//
// Prefill (tensor-core) layout: for every expert x, 256-row unit m and
// 64-wide K block kb, one contiguous chunk of kCodeChunk bytes that a single
// bulk copy brings into shared memory:
//   bytes [0, 8192)     : 256 rows x 8 words of codes; in each 32-bit word the
//                         code of K index 2j sits at bits 4j..4j+3 and the
//                         code of K index 2j+1 at bits 16+4j..16+4j+3 (so the
//                         pair (2j, 2j+1) comes out of one shift and mask as
//                         the two halves of an fp16x2)
//   bytes [8192, 9216)  : 256 rows x (scale fp16 | bias fp16 << 16)
// Gate/up unit m holds gate rows m*128..m*128+127 then up rows of the same
// features; down unit m holds output rows m*256..m*256+255.
// Router prefill layout: unit m (experts m*256..m*256+255, zero rows past E),
// block kb: two 128 x 64 bf16 tiles in the 128-byte swizzled K-major order of
// the tensor-core operand (16-byte chunk c of row r stored at chunk c ^ (r%8)).
//
// Scale and bias: the kernels read one 32-bit word per row and 64-wide K
// block (fp16 scale | fp16 bias << 16).  The caller's pairs may cover groups
// of any multiple of 64 along K (each pair is repeated over its blocks, which
// is exact) and may be bf16: bf16 -> fp16 is exact for 0 and for magnitudes
// 2^-17 .. 65504 (fp16 keeps bf16's 8 significant bits there); a finite value
// that does not survive the conversion sets a flag on which moe_create
// refuses the weights.
//
// Decode layout: one array over all experts (shared expert last) in which
// everything a CTA reads for a run of features is contiguous, so that one
// bulk copy brings it in.  Gate/up: per expert, per feature f, one unit of
// d + d/8 bytes = gate codes of row f (d/2) | up codes of row I+f (d/2) |
// gate scale/bias (d/64 words) | up scale/bias (d/64 words), a word being
// fp16 scale | fp16 bias << 16.  Down: by blocks of 32 input features, for
// each output row the block's 16 bytes of codes (all rows of a block
// contiguous), then the rows' scale/bias words per input group of 64.  Codes
// keep their canonical nibble order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {
namespace {

struct ExpertSrc {
  const uint8_t* codes;
  const uint16_t* scale;
  const uint16_t* bias;
  const uint8_t* sh_codes;
  const uint16_t* sh_scale;
  const uint16_t* sh_bias;
  int E;
  int R;  // rows per expert
  int K;  // inner size
  int group;  // quantisation group along K (a multiple of 64)
  int bf16;   // scale/bias are bf16 (else fp16)
  int* bad;   // kRepackScaleInexact set here when a bf16 value has no exact fp16
};

// 16-bit scale or bias as fp16 bits
__device__ __forceinline__ uint32_t f16_bits(const ExpertSrc& s, uint16_t v) {
  if (!s.bf16) return v;
  const float f = __uint_as_float((uint32_t)v << 16);
  const __half h = __float2half_rn(f);
  if (f == f && __half2float(h) != f) atomicOr(s.bad, kRepackScaleInexact);
  return __half_as_ushort(h);
}

// kernel word of row `row`, 64-wide K block `kb` (fp16 scale | fp16 bias << 16)
__device__ __forceinline__ uint32_t sb_word(const ExpertSrc& s, const uint16_t* sc,
                                            const uint16_t* bi, int row, int kb) {
  const long long gi = (long long)row * (s.K / s.group) + kb / (s.group / 64);
  return f16_bits(s, sc[gi]) | (f16_bits(s, bi[gi]) << 16);
}

__device__ __forceinline__ void expert_ptrs(const ExpertSrc& s, int x, const uint8_t*& c,
                                            const uint16_t*& sc, const uint16_t*& bi) {
  if (x < s.E) {
    c = s.codes + (long long)x * s.R * (s.K / 2);
    sc = s.scale + (long long)x * s.R * (s.K / s.group);
    bi = s.bias + (long long)x * s.R * (s.K / s.group);
  } else {
    c = s.sh_codes;
    sc = s.sh_scale;
    bi = s.sh_bias;
  }
}

__device__ __forceinline__ uint32_t permute_word(uint32_t w) {
  uint32_t o = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t b = (w >> (8 * j)) & 0xFFu;
    o |= (b & 0xFu) << (4 * j);
    o |= (b >> 4) << (16 + 4 * j);
  }
  return o;
}

// gate_up != 0: unit rows = gate m*128.. then up I + m*128..; else rows m*256..
__global__ void repack_prefill_kernel(ExpertSrc s, int nexp, int MU, int gate_up, int I,
                                      uint8_t* __restrict__ out) {
  const int KB = s.K / 64;
  const long long total = (long long)nexp * MU * KB * 256;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(it & 255);
    long long rest = it >> 8;
    const int kb = (int)(rest % KB);
    rest /= KB;
    const int m = (int)(rest % MU);
    const int x = (int)(rest / MU);
    int row;
    if (gate_up) row = (r < 128) ? m * 128 + r : I + m * 128 + (r - 128);
    else row = m * 256 + r;
    const uint8_t* c;
    const uint16_t *sc, *bi;
    expert_ptrs(s, x, c, sc, bi);
    const uint4* src = reinterpret_cast<const uint4*>(c + (long long)row * (s.K / 2) + kb * 32);
    const uint4 a = src[0], b = src[1];
    uint8_t* chunk = out + (((long long)x * MU + m) * KB + kb) * kCodeChunk;
    uint4* dst = reinterpret_cast<uint4*>(chunk + r * 32);
    dst[0] = make_uint4(permute_word(a.x), permute_word(a.y), permute_word(a.z), permute_word(a.w));
    dst[1] = make_uint4(permute_word(b.x), permute_word(b.y), permute_word(b.z), permute_word(b.w));
    reinterpret_cast<uint32_t*>(chunk + 8192)[r] = sb_word(s, sc, bi, row, kb);
  }
}

__global__ void repack_router_prefill_kernel(const uint16_t* __restrict__ wr, int E, int d, int MU,
                                             uint8_t* __restrict__ out) {
  const int KB = d / 64;
  const long long total = (long long)MU * KB * 256 * 8;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(it & 7);
    const int r = (int)((it >> 3) & 255);
    const long long rest = it >> 11;
    const int kb = (int)(rest % KB);
    const int m = (int)(rest / KB);
    const int e = m * 256 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (e < E) v = *reinterpret_cast<const uint4*>(wr + (long long)e * d + kb * 64 + c * 8);
    uint8_t* chunk = out + ((long long)m * KB + kb) * kRouterChunk;
    *reinterpret_cast<uint4*>(chunk + (r >> 7) * 16384 + (r & 127) * 128 + ((c ^ (r & 7)) << 4)) =
        v;
  }
}

// decode gate/up units: thread per 16-byte piece of a unit
__global__ void repack_decode_gu_kernel(ExpertSrc s, int nexp, int I, uint8_t* __restrict__ out) {
  const int d = s.K, ng = d / 64;
  const int ub = d + d / 8;
  const long long pieces = (long long)nexp * I * (ub / 16);
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < pieces;
       it += (long long)gridDim.x * blockDim.x) {
    const long long unit = it / (ub / 16);
    const int o = (int)(it - unit * (ub / 16)) * 16;
    const int x = (int)(unit / I), f = (int)(unit - (long long)x * I);
    const uint8_t* c;
    const uint16_t *sc, *bi;
    expert_ptrs(s, x, c, sc, bi);
    uint4 v;
    if (o < d) {
      const int row = (o < d / 2) ? f : I + f;
      const int off = (o < d / 2) ? o : o - d / 2;
      v = *reinterpret_cast<const uint4*>(c + (long long)row * (d / 2) + off);
    } else {
      const int w = (o - d) / 4;  // first of four words
      const int row = (w < ng) ? f : I + f;
      const int g = (w < ng) ? w : w - ng;
      v = make_uint4(sb_word(s, sc, bi, row, g), sb_word(s, sc, bi, row, g + 1),
                     sb_word(s, sc, bi, row, g + 2), sb_word(s, sc, bi, row, g + 3));
    }
    *reinterpret_cast<uint4*>(out + unit * ub + o) = v;
  }
}

// decode down weights, by blocks of 32 input features: codes
// [x][blk][f] (16 bytes: the block's 32 codes of output row f, canonical
// nibble order), then scale/bias words [x][g][f] (row f, input group g); one
// thread per 16-byte piece of codes or per word
__global__ void repack_decode_dn_kernel(ExpertSrc s, int nexp, uint8_t* __restrict__ out) {
  const int d = s.R, I = s.K, ng = I / 64, nblk = I / 32;
  const long long pieces = (long long)nexp * nblk * d;
  const long long words = (long long)nexp * ng * d;
  uint32_t* sb_out = reinterpret_cast<uint32_t*>(out + pieces * 16);
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < pieces + words;
       it += (long long)gridDim.x * blockDim.x) {
    const uint8_t* c;
    const uint16_t *sc, *bi;
    if (it < pieces) {
      const int f = (int)(it % d);
      const long long xb = it / d;
      const int blk = (int)(xb % nblk), x = (int)(xb / nblk);
      expert_ptrs(s, x, c, sc, bi);
      reinterpret_cast<uint4*>(out)[it] =
          *reinterpret_cast<const uint4*>(c + (long long)f * (I / 2) + blk * 16);
    } else {
      const long long w = it - pieces;
      const int f = (int)(w % d);
      const long long xg = w / d;
      const int g = (int)(xg % ng), x = (int)(xg / ng);
      expert_ptrs(s, x, c, sc, bi);
      sb_out[w] = sb_word(s, sc, bi, f, g);
    }
  }
}

// decode router layout: [d][Ep] bf16, Ep = round_up(E + 1, 8); row f holds
// W_r[0..E-1][f], then w_sg[f], then zeros (16-byte rows: one bulk copy takes
// a CTA's range of rows)
__global__ void repack_router_decode_kernel(const uint16_t* __restrict__ wr,
                                            const uint16_t* __restrict__ wsg, int E, int d,
                                            int Ep, uint16_t* __restrict__ out) {
  const long long total = (long long)d * Ep;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int f = (int)(it / Ep);
    const int e = (int)(it - (long long)f * Ep);
    uint16_t v = 0;
    if (e < E) v = wr[(long long)e * d + f];
    else if (e == E && wsg) v = wsg[f];
    out[it] = v;
  }
}

ExpertSrc make_src(const moe_weights* w, const moe_config& c, bool gu, int* bad) {
  ExpertSrc s;
  s.E = c.E;
  s.group = c.group;
  s.bf16 = c.scale_dtype == MOE_SCALE_BF16;
  s.bad = bad;
  if (gu) {
    s.codes = (const uint8_t*)w->gu_codes;
    s.scale = (const uint16_t*)w->gu_scale;
    s.bias = (const uint16_t*)w->gu_bias;
    s.sh_codes = (const uint8_t*)w->sh_gu_codes;
    s.sh_scale = (const uint16_t*)w->sh_gu_scale;
    s.sh_bias = (const uint16_t*)w->sh_gu_bias;
    s.R = 2 * c.I;
    s.K = c.d;
  } else {
    s.codes = (const uint8_t*)w->dn_codes;
    s.scale = (const uint16_t*)w->dn_scale;
    s.bias = (const uint16_t*)w->dn_bias;
    s.sh_codes = (const uint8_t*)w->sh_dn_codes;
    s.sh_scale = (const uint16_t*)w->sh_dn_scale;
    s.sh_bias = (const uint16_t*)w->sh_dn_bias;
    s.R = c.d;
    s.K = c.I;
  }
  return s;
}

}  // namespace

cudaError_t launch_repack(Handle* h, const moe_weights* w, cudaStream_t st) {
  const moe_config& c = h->cfg;
  const int grid = h->num_sms * 8;
  const ExpertSrc gu = make_src(w, c, true, h->dev_err);
  const ExpertSrc dn = make_src(w, c, false, h->dev_err);
  cudaError_t e = cudaSuccess;
  const dim3 G(grid), B(256);
  if (h->layouts & MOE_LAYOUT_PREFILL) {
    if ((e = launch_kernel(repack_prefill_kernel, G, B, 0, st, gu, h->n_exp, c.I / 128, 1, c.I,
                           h->pf_gu)) != cudaSuccess ||
        (e = launch_kernel(repack_prefill_kernel, G, B, 0, st, dn, h->n_exp, c.d / 256, 0, c.I,
                           h->pf_dn)) != cudaSuccess ||
        (e = launch_kernel(repack_router_prefill_kernel, G, B, 0, st, (const uint16_t*)w->w_router,
                           c.E, c.d, (c.E + 255) / 256, h->pf_router)) != cudaSuccess)
      return e;
  }
  if (h->layouts & MOE_LAYOUT_DECODE) {
    if ((e = launch_kernel(repack_decode_gu_kernel, G, B, 0, st, gu, h->n_exp, c.I, h->dc_gu)) !=
            cudaSuccess ||
        (e = launch_kernel(repack_decode_dn_kernel, G, B, 0, st, dn, h->n_exp, h->dc_dn)) !=
            cudaSuccess ||
        (e = launch_kernel(repack_router_decode_kernel, G, B, 0, st, (const uint16_t*)w->w_router,
                           c.has_shared ? (const uint16_t*)w->w_shared_gate : nullptr, c.E, c.d,
                           decode_router_pitch(c.E), h->dc_router_t)) != cudaSuccess)
      return e;
  }
  e = cudaMemcpyAsync(h->w_router, w->w_router, (size_t)c.E * c.d * 2, cudaMemcpyDeviceToDevice,
                      st);
  if (e != cudaSuccess) return e;
  if (c.has_shared)
    return cudaMemcpyAsync(h->w_sg, w->w_shared_gate, (size_t)c.d * 2, cudaMemcpyDeviceToDevice,
                           st);
  return cudaMemsetAsync(h->w_sg, 0, (size_t)c.d * 2, st);
}

}  // namespace moe
