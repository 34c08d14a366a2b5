// Top-k of one token's expert logits by one warp, for up to 256 experts.
// Source: Perplexity, "Optimizing on-device inference for Apple Silicon",
// §"Qwen creates three different workload shapes" (the router keeps 8 of 256
// experts per token).  Ranking: logit descending, then expert index
// ascending.
//
// Lane l holds the 64-bit keys of experts 8l .. 8l+7 in s[0..7]: key =
// order key of the logit (ord_key) << 32 | (0xFFFFFFFF - e), 0 where there is
// no expert; distinct keys, larger is better.  The lane sorts its eight keys
// descending (Batcher's 19-comparator network), then k rounds: the largest
// list head over the warp (a warp maximum of the heads' high words; among
// equal logits the lowest lane holds the lowest expert index, and within a
// lane the sorted order already puts it first), whose lane drops it.  A lane
// holds eight experts, so it wins at most eight rounds; k <= 32.
#pragma once
#include <cstdint>

namespace moe {

// order-preserving key of a float (larger value, larger key); -0 taken as +0
__device__ __forceinline__ uint32_t ord_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// the float of an order key (ord_key's inverse; -0 comes back as +0)
__device__ __forceinline__ float ord_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Returns, in lane r < k, the key of the expert of rank r (0 in the other
// lanes); the expert is 0xFFFFFFFF - (uint32_t)key, the logit
// ord_value(key >> 32).  s is destroyed.
__device__ __forceinline__ unsigned long long warp_topk_lists(unsigned long long (&s)[8], int k,
                                                              int lane) {
#define MOE_CE(a, b)                               \
  {                                                \
    const unsigned long long x_ = s[a], y_ = s[b]; \
    const bool sw_ = x_ < y_;                      \
    s[a] = sw_ ? y_ : x_;                          \
    s[b] = sw_ ? x_ : y_;                          \
  }
  MOE_CE(0, 1) MOE_CE(2, 3) MOE_CE(4, 5) MOE_CE(6, 7)
  MOE_CE(0, 2) MOE_CE(1, 3) MOE_CE(4, 6) MOE_CE(5, 7)
  MOE_CE(1, 2) MOE_CE(5, 6)
  MOE_CE(0, 4) MOE_CE(1, 5) MOE_CE(2, 6) MOE_CE(3, 7)
  MOE_CE(2, 4) MOE_CE(3, 5)
  MOE_CE(1, 2) MOE_CE(3, 4) MOE_CE(5, 6)
#undef MOE_CE
  unsigned long long mine = 0ull;
  for (int r = 0; r < k; ++r) {
    const uint32_t hi = (uint32_t)(s[0] >> 32);
    const uint32_t m = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t bal = __ballot_sync(0xffffffffu, hi == m);
    const bool win = (bal & ((2u << lane) - 1u)) == (1u << lane);  // lowest lane with m
    const unsigned long long kw = __shfl_sync(0xffffffffu, s[0], __ffs(bal) - 1);
    if (lane == r) mine = kw;
#pragma unroll
    for (int i = 0; i < 7; ++i) s[i] = win ? s[i + 1] : s[i];
    s[7] = win ? 0ull : s[7];
  }
  return mine;
}

}  // namespace moe
