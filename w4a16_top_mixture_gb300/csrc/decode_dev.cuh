// Device helpers shared by the fused decode kernels: the compile-time block shape, warp reductions, the
// lane order of routed h vectors, and the two inner loops every decode kernel runs -- the dot products of
// quantised rows with fp16 activations (dot_rows) and the warp top-k over one token's expert logits.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;

constexpr size_t c_align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Compile-time block shape: every width, stride and loop bound of the decode kernel is a constant, which keeps
// its machine code small (the kernel's executed code must stay resident in the SM instruction cache).
template <int H_, int E_, int K_, int I_, int Is_>
struct Shape {
  static constexpr int H = H_, E = E_, K = K_, I = I_, Is = Is_;
  static constexpr int GB = H / 64, GI = I / 64, GS = Is / 64;
  static constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  static constexpr size_t RR = c_align16((size_t)H + (size_t)GB * 4);
  static constexpr size_t SU = c_align16(2 * (size_t)H + 2 * (size_t)GB * 4);
  static constexpr size_t SDR = c_align16((size_t)Is + (size_t)GS * 4);
  static constexpr size_t EU = c_align16((size_t)H + 2 * (size_t)GB * 4);
  static constexpr size_t DR = c_align16((size_t)I / 2 + (size_t)GI * 4);
  static constexpr size_t exgu_expert = (size_t)I * EU;
  static constexpr size_t exdn_expert = (size_t)H * DR;
};
using ShapeProd = Shape<2048, 256, 8, 512, 512>;
using ShapeTiny = Shape<512, 32, 4, 128, 128>;

__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)(((unsigned)n * (unsigned)c) / (unsigned)G); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}


template <int NR, int TK>
struct DotR {
  float v[TK][NR];
};

// Routed h vectors are stored in the lane order of the down dot: unit u = 16 c + 4 j + m (lane chunk c,
// float4 j, component m) sits at float index (j * (I/16) + c) * 4 + m, so that a linear copy of a vector into
// shared memory lets lane c read its float4 j at consecutive 16-byte addresses across the warp.
template <int I>
__device__ __forceinline__ int hpos(int u) {
  return (((u & 15) >> 2) * (I / 16) + (u >> 4)) * 4 + (u & 3);
}

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ---- integer dot products (dp2a) on 16-bit fixed-point activations
//
// Activations enter the dot products as int16 values with a power-of-two scale per block of columns (a 32-column
// chunk of x, or a lane's 16 values of h): v = 2^-sc * q, |q| <= 32767, the scale chosen from the block's
// largest magnitude. Every fp16 input in the block's top five binades is represented exactly; smaller ones are
// rounded to the block's grid. Weight codes enter as they are stored (unsigned bytes, or nibbles masked in
// place), so every product and every partial sum over a block is exact in int32; the group's affine is then
// applied once per block in fp32: sum_c (s q_c + b) v_c = 2^-sc (s * sum_c q_c a_c + b * sum_c a_c).
//
// Code layouts that these routines read (written at load time):
//   int8 rows: every 8-byte block holds columns 0 1 4 5 2 3 6 7;
//   int4 rows: every 32-bit word holds columns 0..7 as bytes (c0|c2<<4, c1|c3<<4, c4|c6<<4, c5|c7<<4);
// so that both deliver the column pairs (0,1) (4,5) (2,3) (6,7) to the four dp2a of a block, and the
// activations of 8 columns are one uint4 of int16 pairs in that order.

// d = c + a.h0 * b.b0 + a.h1 * b.b1 (lo) or + a.h0 * b.b2 + a.h1 * b.b3 (hi); a signed 16-bit, b unsigned bytes
__device__ __forceinline__ int dp2lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One 8-column block of codes against one uint4 of activation pairs. int4: word w, the low nibbles accumulate
// into lo, the high nibbles (kept in place, i.e. times 16) into hi; int8: words w0, w1.
__device__ __forceinline__ void dp_int4(uint32_t w, const uint4& x, int& lo, int& hi) {
  const uint32_t l = w & 0x0F0F0F0Fu, h = w & 0xF0F0F0F0u;
  lo = dp2lo(x.x, l, lo);
  lo = dp2hi(x.y, l, lo);
  hi = dp2lo(x.z, h, hi);
  hi = dp2hi(x.w, h, hi);
}
__device__ __forceinline__ int dp_int8(uint32_t w0, uint32_t w1, const uint4& x, int acc) {
  acc = dp2lo(x.x, w0, acc);
  acc = dp2hi(x.y, w0, acc);
  acc = dp2lo(x.z, w1, acc);
  return dp2hi(x.w, w1, acc);
}

// Power-of-two scale for a block whose largest magnitude is m: sc = 2^(15 - e) with m < 2^e, so |v * sc| <
// 32768; inv = 1 / sc. Read from the exponent bits (exact; blocks of zeros or tiny values use the smallest e).
__device__ __forceinline__ void block_scale(float m, float& sc, float& inv) {
  uint32_t E = (__float_as_uint(m) >> 23) & 0xFFu;
  E = E < 15u ? 15u : E;
  sc = __uint_as_float((268u - E) << 23);
  inv = __uint_as_float((E - 14u) << 23);
}
__device__ __forceinline__ int q16(float v, float sc) {
  const int q = __float2int_rn(v * sc);
  return q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
}
__device__ __forceinline__ uint32_t pk16(int a, int b) { return (uint32_t)(a & 0xFFFF) | ((uint32_t)b << 16); }

// 8 consecutive values -> the uint4 of int16 pairs (0,1) (4,5) (2,3) (6,7); returns their integer sum
__device__ __forceinline__ int quant8(const float* v, float sc, uint4& o) {
  int q[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) q[k] = q16(v[k], sc);
  o.x = pk16(q[0], q[1]);
  o.y = pk16(q[4], q[5]);
  o.z = pk16(q[2], q[3]);
  o.w = pk16(q[6], q[7]);
  return ((q[0] + q[1]) + (q[2] + q[3])) + ((q[4] + q[5]) + (q[6] + q[7]));
}

// A lane's 16 consecutive values of an fp32 vector (h of a routed expert, hs of the shared one) as int16 pairs
// for the down projections: p[0] covers columns 0..7, p[1] columns 8..15; inv and the integer sum for the fold.
struct Act16 {
  uint4 p[2];
  float inv;
  float sum;   // inv * sum of the integers
};
__device__ __forceinline__ Act16 quant_lane16(float4 h0, float4 h1, float4 h2, float4 h3) {
  const float v[16] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w, h2.x, h2.y, h2.z, h2.w, h3.x, h3.y, h3.z, h3.w};
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(v[k]));
  Act16 a;
  float sc;
  block_scale(m, sc, a.inv);
  const int s = quant8(v, sc, a.p[0]) + quant8(v + 8, sc, a.p[1]);
  a.sum = (float)s * a.inv;
  return a;
}

// One lane's 16 columns of a routed down row (int4, two words) or of a shared down row (int8, 16 bytes) against
// its quantised activation: the group's affine folded in, s * sum(q v) + b * sum(v).
__device__ __forceinline__ float down_int4(uint2 w, float2 sb, const Act16& a) {
  int lo = 0, hi = 0;
  dp_int4(w.x, a.p[0], lo, hi);
  dp_int4(w.y, a.p[1], lo, hi);
  return sb.x * ((float)(lo + (hi >> 4)) * a.inv) + sb.y * a.sum;
}
__device__ __forceinline__ float down_int8(uint4 w, float2 sb, const Act16& a) {
  int acc = dp_int8(w.x, w.y, a.p[0], 0);
  acc = dp_int8(w.z, w.w, a.p[1], acc);
  return sb.x * ((float)acc * a.inv) + sb.y * a.sum;
}

// Dot products of NR rows (a warp's work item) with up to TK tokens. INT8 = false: int4 rows (32 codes of a
// chunk = 16 bytes at chunk * 16); INT8 = true: lane-interleaved int8 rows (16-byte halves of chunk c = l + LW*p
// at ((2p + half) * LW + l) * 16). Lane l covers the 32-column chunks c = l + LW*p. Activations: x16[((t*P + p)*4
// + j)*LW + l] the uint4 of 8-column block j of chunk c for token t; xsc[(t*P + p)*LW + l] = (inv, sum of the
// chunk's quantised values times inv). Only the chunks of p in [p0, p1) are covered (p1 < 0: every p), so that
// warps can share a row. Returns the warp-reduced v[tt][r] in every lane. Inlined: an out-of-line
// call would save and restore the caller's registers through local memory, which has almost no L1 behind it when
// shared memory takes the whole carveout.
template <int H, int NR, int TK, bool INT8>
__device__ __forceinline__ DotR<NR, TK> dot_rows(const uint8_t* r0, const uint8_t* r1, const uint8_t* r2,
                                              const uint8_t* r3, const uint8_t* s0, const uint8_t* s1,
                                              const uint8_t* s2, const uint8_t* s3, int nvalid,
                                              const uint4* __restrict__ x16, const float2* __restrict__ xsc,
                                              int ta, int tb, int nt, int p0 = 0, int p1 = -1) {
  constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  const int lane = threadIdx.x & 31;
  const uint8_t* rp[4] = {r0, r1, r2, r3};
  const uint8_t* sp[4] = {s0, s1, s2, s3};
  int tix[TK];
  tix[0] = ta;
  if (TK > 1) tix[TK - 1] = tb;
  DotR<NR, TK> out;
#pragma unroll
  for (int tt = 0; tt < TK; ++tt)
#pragma unroll
    for (int r = 0; r < NR; ++r) out.v[tt][r] = 0.f;
  if (lane < LW) {
#pragma unroll 1
    for (int p = p0; p < (p1 < 0 ? P : p1); ++p) {
      const int c = lane + LW * p;
      int lo[TK][NR], hi[TK][NR];
#pragma unroll
      for (int tt = 0; tt < TK; ++tt)
#pragma unroll
        for (int r = 0; r < NR; ++r) lo[tt][r] = hi[tt][r] = 0;
      uint4 ca[NR], cb[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (INT8) {
          ca[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + ((p * 2) * LW + lane) * 16) : make_uint4(0, 0, 0, 0);
          cb[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + ((p * 2 + 1) * LW + lane) * 16) : make_uint4(0, 0, 0, 0);
        } else {
          ca[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + c * 16) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // 8-column block j of the chunk
        uint4 xv[TK];
#pragma unroll
        for (int tt = 0; tt < TK; ++tt)
          xv[tt] = tt < nt ? x16[((tix[tt] * P + p) * 4 + j) * LW + lane] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
          for (int tt = 0; tt < TK; ++tt) {
            if (INT8) {
              const uint4& q4 = j < 2 ? ca[r] : cb[r];
              lo[tt][r] = dp_int8((j & 1) ? q4.z : q4.x, (j & 1) ? q4.w : q4.y, xv[tt], lo[tt][r]);
            } else {
              dp_int4(j == 0 ? ca[r].x : j == 1 ? ca[r].y : j == 2 ? ca[r].z : ca[r].w, xv[tt], lo[tt][r],
                      hi[tt][r]);
            }
          }
        }
      }
      // the group's affine on the chunk's exact integer sums
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < nvalid) {
          const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(sp[r] + (c >> 1) * 4));
#pragma unroll
          for (int tt = 0; tt < TK; ++tt) {
            const float2 X = tt < nt ? xsc[(tix[tt] * P + p) * LW + lane] : make_float2(0.f, 0.f);
            const int a = INT8 ? lo[tt][r] : lo[tt][r] + (hi[tt][r] >> 4);
            out.v[tt][r] += sb.x * ((float)a * X.x) + sb.y * X.y;
          }
        }
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < TK; ++tt)
#pragma unroll
    for (int r = 0; r < NR; ++r) out.v[tt][r] = warp_sum(out.v[tt][r]);
  return out;
}

// The x prologue of a decode kernel: one 8-column block of a 32-column chunk, quantised into x16 / xsc (see
// dot_rows). The four threads of a chunk (blocks j = 0..3) are consecutive lanes of one warp, and all 32 lanes
// of the warp call this together (live = false for lanes without a block): the chunk's largest magnitude and
// integer sum are reduced over the four lanes. v: the block's 8 values (already RMS-normalised in the stacked
// layer).
template <int LW, int P>
__device__ __forceinline__ void quant_block8(const float* v, bool live, int t, int c, int j, uint4* x16,
                                             float2* xsc) {
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
  m = fmaxf(m, __shfl_xor_sync(FULL, m, 1));
  m = fmaxf(m, __shfl_xor_sync(FULL, m, 2));
  float sc, inv;
  block_scale(m, sc, inv);
  uint4 o;
  int s = quant8(v, sc, o);
  s += __shfl_xor_sync(FULL, s, 1);
  s += __shfl_xor_sync(FULL, s, 2);
  if (live) {
    const int l = c % LW, p = c / LW;
    x16[((t * P + p) * 4 + j) * LW + l] = o;
    if (j == 0) xsc[(t * P + p) * LW + l] = make_float2(inv, (float)s * inv);
  }
}



}  // namespace
}  // namespace moe
