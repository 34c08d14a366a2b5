// Device implementation of the seeded input generator of synth/gen.py (the
// same counter-based definition, bit for bit): SplitMix64 output function
// (Steele, Lea & Flood, OOPSLA 2014) on counters, Irwin-Hall sum of eight
// 16-bit uniforms times one fp32 constant, round-to-nearest-even to bf16,
// and the group-affine 4-bit quantiser.  Inputs only: nothing here computes
// any part of the MoE block.  Every arithmetic step is an explicitly rounded
// IEEE operation (no contraction into FMA), so the host and the device agree.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float normal_value(uint64_t key, uint64_t n, float c) {
  const uint64_t a = mix64(key + (2 * n + 1) * kGamma);
  const uint64_t b = mix64(key + (2 * n + 2) * kGamma);
  long long s = 0;
#pragma unroll
  for (int sh = 0; sh < 64; sh += 16) s += (long long)((a >> sh) & 0xFFFFull) + (long long)((b >> sh) & 0xFFFFull);
  const float z = (float)(s - 262140ll);  // exact: |z| < 2^19
  return __fmul_rn(z, c);
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float v) {
  uint32_t u = __float_as_uint(v);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t start, uint64_t count, float c,
                                   uint16_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = bf16_rne_bits(normal_value(key, start + i, c));
}

// one thread per (row, group of 64)
__global__ void quantized_kernel(uint64_t key, int rows, int K, float c, uint8_t* codes,
                                 uint16_t* scale, uint16_t* bias) {
  const int G = K / 64;
  const long long total = (long long)rows * G;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long row = it / G;
    const int g = (int)(it - row * G);
    const uint64_t n0 = (uint64_t)row * K + (uint64_t)g * 64;
    float w[64];
    float mn = 0.f, mx = 0.f;
#pragma unroll 8
    for (int i = 0; i < 64; ++i) {
      w[i] = normal_value(key, n0 + i, c);
      mn = (i == 0 || w[i] < mn) ? w[i] : mn;
      mx = (i == 0 || w[i] > mx) ? w[i] : mx;
    }
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
    const __half b16 = __float2half_rn(mn);
    const float s = __half2float(s16), b = __half2float(b16);
    uint8_t* out = codes + row * (K / 2) + g * 32;
#pragma unroll 8
    for (int i = 0; i < 64; i += 2) {
      int q0 = 0, q1 = 0;
      if (s != 0.f) {
        q0 = (int)rintf(__fdiv_rn(__fsub_rn(w[i], b), s));
        q1 = (int)rintf(__fdiv_rn(__fsub_rn(w[i + 1], b), s));
        q0 = q0 < 0 ? 0 : (q0 > 15 ? 15 : q0);
        q1 = q1 < 0 ? 0 : (q1 > 15 ? 15 : q1);
      }
      out[i / 2] = (uint8_t)(q0 | (q1 << 4));
    }
    scale[it] = __half_as_ushort(s16);
    bias[it] = __half_as_ushort(b16);
  }
}

}  // namespace

extern "C" {

int synth_normal_bf16(uint64_t key, uint64_t start, uint64_t count, float c, void* out,
                      void* stream) {
  if (count == 0) return 0;
  normal_bf16_kernel<<<1024, 256, 0, (cudaStream_t)stream>>>(key, start, count, c,
                                                             (uint16_t*)out);
  return (int)cudaGetLastError();
}

int synth_quantized(uint64_t key, int rows, int K, float c, void* codes, void* scale, void* bias,
                    void* stream) {
  if (rows <= 0) return 0;
  quantized_kernel<<<1024, 128, 0, (cudaStream_t)stream>>>(key, rows, K, c, (uint8_t*)codes,
                                                           (uint16_t*)scale, (uint16_t*)bias);
  return (int)cudaGetLastError();
}

}
