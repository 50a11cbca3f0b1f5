// Inline-PTX helpers for sm_103a: mbarriers, 1-D bulk async copies (TMA engine), globaltimer, and the code
// unpacking used by every dot product. Unpacking relies only on IEEE-754 encoding facts:
//   * a float whose exponent field is that of 2^23 and whose low mantissa bits hold an integer v (< 2^23) is
//     exactly 2^23 + v, so OR-ing a code field into 0x4B000000 in place and removing 2^23 by an exact fused
//     multiply-add recovers the code as a float with no integer-to-float conversion;
//   * codes left at bit position 4k (or 8k) come out multiplied by 2^(4k) (2^(8k)); the same fused step
//     multiplies by the exact power of two 2^-4k (2^-8k).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// orders this thread's earlier generic-proxy view of global memory before its later async-proxy (bulk copy)
// reads of global memory
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase completes (or the hint
// elapses) instead of spinning, so idle warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false if the phase did not complete within timeout_ns. The loop is kept out of line
// so that the many call sites share one copy of it (instruction-cache footprint).
__device__ __forceinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (globaltimer() - t0 > timeout_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, timeout_ns);
}
// 1-D bulk copy global -> shared through the TMA engine, completing on an mbarrier (transaction bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Bulk prefetch of a global range into L2 (no destination, no completion tracking).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded spin until *cnt >= target. Returns false on timeout.
__device__ __forceinline__ bool spin_geq(const uint32_t* cnt, uint32_t target, uint64_t timeout_ns) {
  if (ld_acquire_u32(cnt) >= target) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 8; ++i) {
      if (ld_acquire_u32(cnt) >= target) return true;
      __nanosleep(20);
    }
    if (globaltimer() - t0 > timeout_ns) return false;
  }
}

constexpr uint32_t MAGIC = 0x4B000000u;   // bit pattern of 2^23

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float bits(uint32_t v) { return __uint_as_float(v); }

// One 32-bit word of int4 codes (element n of the word in bits 4n..4n+3) -> the pairs
// (q_k, q_{4+k}) for k = 0..3, exact, as floats.
__device__ __forceinline__ void unpack_int4_word(uint32_t w, float2 q[4]) {
  const uint32_t hi = w >> 16;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t m = 0xFu << (4 * k);
    const float sc = __uint_as_float((uint32_t)(127 - 4 * k) << 23);            // 2^-4k
    const float off = -__uint_as_float((uint32_t)(127 + 23 - 4 * k) << 23);     // -2^(23-4k)
    q[k] = __ffma2_rn(f2(bits((w & m) | MAGIC), bits((hi & m) | MAGIC)), f2(sc, sc), f2(off, off));
  }
}

// Two 32-bit words of int8 codes (columns 0..3 in w0, 4..7 in w1, column n in byte n%4) -> the pairs
// (q_k, q_{4+k}) for k = 0..3, exact.
__device__ __forceinline__ void unpack_int8_pair(uint32_t w0, uint32_t w1, float2 q[4]) {
  const uint32_t h0 = w0 >> 16, h1 = w1 >> 16;
  const float s8 = __uint_as_float((uint32_t)(127 - 8) << 23);          // 2^-8
  const float o0 = -8388608.0f;                                         // -2^23
  const float o8 = -__uint_as_float((uint32_t)(127 + 15) << 23);        // -2^15
  q[0] = __ffma2_rn(f2(bits((w0 & 0xFFu) | MAGIC), bits((w1 & 0xFFu) | MAGIC)), f2(1.f, 1.f), f2(o0, o0));
  q[1] = __ffma2_rn(f2(bits((w0 & 0xFF00u) | MAGIC), bits((w1 & 0xFF00u) | MAGIC)), f2(s8, s8), f2(o8, o8));
  q[2] = __ffma2_rn(f2(bits((h0 & 0xFFu) | MAGIC), bits((h1 & 0xFFu) | MAGIC)), f2(1.f, 1.f), f2(o0, o0));
  q[3] = __ffma2_rn(f2(bits((h0 & 0xFF00u) | MAGIC), bits((h1 & 0xFF00u) | MAGIC)), f2(s8, s8), f2(o8, o8));
}

// One 32-bit word of int8 codes (column n in byte n) -> (q0, q1), (q2, q3), exact.
__device__ __forceinline__ void unpack_int8_word(uint32_t w, float2& q01, float2& q23) {
  const uint32_t h = w >> 16;
  const float s8 = 0.00390625f;
  q01 = __ffma2_rn(f2(bits((w & 0xFFu) | MAGIC), bits((w & 0xFF00u) | MAGIC)), f2(1.f, s8), f2(-8388608.0f, -32768.0f));
  q23 = __ffma2_rn(f2(bits((h & 0xFFu) | MAGIC), bits((h & 0xFF00u) | MAGIC)), f2(1.f, s8), f2(-8388608.0f, -32768.0f));
}

// Four int4 codes of a 16-bit field (columns 4m..4m+3 of a canonically packed int4 row) -> (q0, q1), (q2, q3),
// exact.
__device__ __forceinline__ void unpack_int4_quad(uint32_t hw, float2& q01, float2& q23) {
  const float a = bits((hw & 0xFu) | MAGIC), b = bits((hw & 0xF0u) | MAGIC);
  const float c = bits((hw & 0xF00u) | MAGIC), d = bits((hw & 0xF000u) | MAGIC);
  q01 = __ffma2_rn(f2(a, b), f2(1.f, 0.0625f), f2(-8388608.0f, -524288.0f));
  q23 = __ffma2_rn(f2(c, d), f2(0.00390625f, 0.000244140625f), f2(-32768.0f, -2048.0f));
}

constexpr uint32_t MAGIC16 = 0x64006400u;   // fp16 pair (1024, 1024): codes OR-ed into the low mantissa bits

// f32 += f16 * f16 on the low (or high) halves of two 32-bit registers; the product is exact in fp32.
__device__ __forceinline__ float fmix_lo(uint32_t a, uint32_t b, float c) {
  asm("{\n .reg .f16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.f16 %0, al, bl, %0;\n}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}
__device__ __forceinline__ float fmix_hi(uint32_t a, uint32_t b, float c) {
  asm("{\n .reg .f16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.f16 %0, ah, bh, %0;\n}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// Code pairs as fp16 (1024 + code) values, two per 32-bit register, in the column pairing (k, 4+k) of an
// 8-column block. int4 word w (column n in bits 4n..4n+3): v[0] = (q0, q4), v[2] = (q2, q6) hold 1024 + q;
// v[1] = (q1, q5), v[3] = (q3, q7) hold 1024 + 16 q. int8 block stored as bytes [c0 c1 c4 c5 | c2 c3 c6 c7]
// in words w0, w1: v[0] = (c0, c4), v[1] = (c1, c5), v[2] = (c2, c6), v[3] = (c3, c7), all 1024 + code.
__device__ __forceinline__ void int4_word_pairs(uint32_t w, uint32_t v[4]) {
  const uint32_t w8 = w >> 8;
  v[0] = (w & 0x000F000Fu) | MAGIC16;
  v[1] = (w & 0x00F000F0u) | MAGIC16;
  v[2] = (w8 & 0x000F000Fu) | MAGIC16;
  v[3] = (w8 & 0x00F000F0u) | MAGIC16;
}
__device__ __forceinline__ void int8_block_pairs(uint32_t w0, uint32_t w1, uint32_t v[4]) {
  v[0] = (w0 & 0x00FF00FFu) | MAGIC16;
  v[1] = ((w0 >> 8) & 0x00FF00FFu) | MAGIC16;
  v[2] = (w1 & 0x00FF00FFu) | MAGIC16;
  v[3] = ((w1 >> 8) & 0x00FF00FFu) | MAGIC16;
}

__device__ __forceinline__ float2 h2f(uint32_t sb) {   // packed (s, b) fp16 pair -> floats
  __half2 h = *reinterpret_cast<__half2*>(&sb);
  return __half22float2(h);
}

}  // namespace moe
