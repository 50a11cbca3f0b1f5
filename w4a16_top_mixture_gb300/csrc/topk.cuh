// Warp-wide top-k over a row of router logits, shared by the decode kernels and the chunk path's routing.
#pragma once
#include <stdint.h>

namespace moe {
namespace {

// Top-k of E logits by one warp, without side effects: lane l holds experts l*EPL .. l*EPL+EPL-1 as
// order-preserving integer keys (a real logit's key is at least 1, an entry beyond E and an entry already taken
// have key 0, so K <= E rounds always pick K distinct experts below E, NaN and infinite logits included: NaN ranks
// above +inf); each of the K rounds takes the warp maximum (the lowest lane winning a tie,
// inside a lane the lowest index) and only the winning lane recomputes its maximum. Lane j < K returns the
// j-th largest (index, logit).
// VEC: E == 32 * EPL, EPL a multiple of 4 and lg 16-byte aligned, so every lane reads its logits as whole
// 16-byte words (a row of a [T][E+1] array is aligned only for t = 0).
template <int EPL, bool VEC>
__device__ __forceinline__ void warp_topk_lean(const float* __restrict__ lg, int E, int K, int& my_idx,
                                            float& my_logit) {
  const int lane = threadIdx.x & 31;
  uint32_t key[EPL];
  if (VEC) {
#pragma unroll
    for (int i = 0; i < EPL; i += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(lg + lane * EPL + i));
      const uint32_t b[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)};
#pragma unroll
      for (int k = 0; k < 4; ++k) key[i + k] = max((b[k] & 0x80000000u) ? ~b[k] : (b[k] | 0x80000000u), 1u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      const uint32_t b = e < E ? __float_as_uint(__ldcg(lg + e)) : 0u;
      key[i] = e < E ? max((b & 0x80000000u) ? ~b : (b | 0x80000000u), 1u) : 0u;
    }
  }
  uint32_t best = key[0];
  int bi = 0;
#pragma unroll
  for (int i = 1; i < EPL; ++i)
    if (key[i] > best) { best = key[i]; bi = i; }
  my_idx = -1;
  uint32_t my_key = 0;
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
    const int win = __ffs(__ballot_sync(0xFFFFFFFFu, best == m)) - 1;
    const int sel = __shfl_sync(0xFFFFFFFFu, lane * EPL + bi, win);
    if (lane == j) { my_idx = sel; my_key = m; }
    if (lane == win) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == bi) key[i] = 0u;
      best = key[0];
      bi = 0;
#pragma unroll
      for (int i = 1; i < EPL; ++i)
        if (key[i] > best) { best = key[i]; bi = i; }
    }
  }
  const uint32_t b = (my_key & 0x80000000u) ? (my_key & 0x7FFFFFFFu) : ~my_key;
  my_logit = __uint_as_float(b);
}

}  // namespace
}  // namespace moe
