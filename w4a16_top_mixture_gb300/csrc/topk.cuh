// Warp-wide top-k over a row of router logits, shared by the decode kernels and the chunk path's routing.
#pragma once
#include <stdint.h>

namespace moe {
namespace {

// Order-preserving integer key of a logit, at least 1 (0 marks an entry beyond E or one already taken), and
// back. NaN ranks above +inf.
__device__ __forceinline__ uint32_t topk_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return max((b & 0x80000000u) ? ~b : (b | 0x80000000u), 1u);
}
__device__ __forceinline__ float topk_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// EPL = 8: every lane first sorts its eight (key, index) pairs, larger key first and on equal keys the lower
// index first (a 19-comparator network; any correct network gives this one order, the comparison being total on
// distinct pairs); then each round takes the warp maximum of the lanes' heads and the winning lane shifts its
// list by one, so no round rescans a lane.
__device__ __forceinline__ void topk_cmpx(uint32_t (&k)[8], int (&ix)[8], int a, int b) {
  const bool keep = k[a] > k[b] || (k[a] == k[b] && ix[a] < ix[b]);
  const uint32_t ka = k[a], kb = k[b];
  const int ia = ix[a], ib = ix[b];
  k[a] = keep ? ka : kb;
  k[b] = keep ? kb : ka;
  ix[a] = keep ? ia : ib;
  ix[b] = keep ? ib : ia;
}
__device__ __forceinline__ void warp_topk_sorted8(uint32_t (&key)[8], int K, int& my_idx, uint32_t& my_key) {
  const int lane = threadIdx.x & 31;
  int ix[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ix[i] = lane * 8 + i;
  topk_cmpx(key, ix, 0, 2); topk_cmpx(key, ix, 1, 3); topk_cmpx(key, ix, 4, 6); topk_cmpx(key, ix, 5, 7);
  topk_cmpx(key, ix, 0, 4); topk_cmpx(key, ix, 1, 5); topk_cmpx(key, ix, 2, 6); topk_cmpx(key, ix, 3, 7);
  topk_cmpx(key, ix, 0, 1); topk_cmpx(key, ix, 2, 3); topk_cmpx(key, ix, 4, 5); topk_cmpx(key, ix, 6, 7);
  topk_cmpx(key, ix, 2, 4); topk_cmpx(key, ix, 3, 5);
  topk_cmpx(key, ix, 1, 4); topk_cmpx(key, ix, 3, 6);
  topk_cmpx(key, ix, 1, 2); topk_cmpx(key, ix, 3, 4); topk_cmpx(key, ix, 5, 6);
  my_idx = -1;
  my_key = 0;
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, key[0]);
    const int win = __ffs(__ballot_sync(0xFFFFFFFFu, key[0] == m)) - 1;
    const int sel = __shfl_sync(0xFFFFFFFFu, ix[0], win);
    if (lane == j) { my_idx = sel; my_key = m; }
    if (lane == win) {
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        key[i] = key[i + 1];
        ix[i] = ix[i + 1];
      }
      key[7] = 0u;
    }
  }
}

// Top-k over keys held by one warp: lane l holds experts l*EPL .. l*EPL+EPL-1 (key 0 for entries beyond E).
// K <= E rounds, each taking the warp maximum (the lowest lane winning a tie, inside a lane the lowest index, so
// the lowest index overall), always pick K distinct experts below E, NaN and infinite logits included. Lane
// j < K returns the j-th largest (index, key). The keys are consumed.
// Other EPL: the winning lane of each round rescans its keys.
template <int EPL>
__device__ __forceinline__ void warp_topk_keys(uint32_t (&key)[EPL], int K, int& my_idx, uint32_t& my_key) {
  if constexpr (EPL == 8) {
    warp_topk_sorted8(key, K, my_idx, my_key);
    return;
  }
  const int lane = threadIdx.x & 31;
  uint32_t best = key[0];
  int bi = 0;
#pragma unroll
  for (int i = 1; i < EPL; ++i)
    if (key[i] > best) { best = key[i]; bi = i; }
  my_idx = -1;
  my_key = 0;
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
}

// The same over E logits in global memory (lane l reads experts l*EPL .. l*EPL+EPL-1); lane j < K returns the
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
      key[i] = topk_key(v.x);
      key[i + 1] = topk_key(v.y);
      key[i + 2] = topk_key(v.z);
      key[i + 3] = topk_key(v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      key[i] = e < E ? topk_key(__ldcg(lg + e)) : 0u;
    }
  }
  uint32_t my_key;
  warp_topk_keys<EPL>(key, K, my_idx, my_key);
  my_logit = topk_logit(my_key);
}

}  // namespace
}  // namespace moe
