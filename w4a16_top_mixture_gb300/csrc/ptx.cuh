// Inline-PTX helpers for sm_103a: mbarriers, 1-D bulk async copies (TMA engine), globaltimer, bounded waits,
// and the code-to-fp16 unpacking of the prompt-chunk GEMM. That unpacking relies only on an IEEE-754 encoding
// fact: an fp16 value whose exponent field is that of 1024 and whose low mantissa bits hold an integer v < 1024
// is exactly 1024 + v, so OR-ing a code field into 0x6400 yields 1024 + code (or 1024 + 16 code for a field at
// bit 4) with no integer-to-float conversion.
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
// true in exactly one lane of a converged warp. Work done under it with operands computed by the whole warp
// keeps those operands warp-uniform, which the copy and tensor-core issue instructions take directly.
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile("{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}" : "=r"(p));
  return p != 0;
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
// Bounded wait: returns false if the phase did not complete within timeout_ns. The loop is kept out of line so
// that the many call sites share one copy of it (instruction-cache footprint of the kernels).
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
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
// 64-bit relaxed accesses at GPU scope. A naturally aligned 64-bit access is single-copy atomic, so a word that
// carries a value and a tag is seen whole or not at all (each element of the two-word load on its own).
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void ld_relaxed_u64x2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
// *cnt += v with release semantics at GPU scope: every write this thread made before (and every write it has
// observed, e.g. through a preceding barrier) is visible to a thread that later reads the new count with an
// acquire load (ld_acquire_u32). One instruction in place of a full fence followed by an atomic.
__device__ __forceinline__ void red_release_add(uint32_t* cnt, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(cnt), "r"(v) : "memory");
}

// 64-bit counts that only grow (the single-token kernel's exchange counts, compared with epoch * expected)
__device__ __forceinline__ void red_release_add_u64(uint64_t* cnt, uint64_t v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(cnt), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
static __device__ __noinline__ bool spin_geq_u64_slow(const uint64_t* cnt, uint64_t target, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 8; ++i) {
      if (ld_acquire_u64(cnt) >= target) return true;
      __nanosleep(20);
    }
    if (globaltimer() - t0 > timeout_ns) return false;
  }
}
__device__ __forceinline__ bool spin_geq_u64(const uint64_t* cnt, uint64_t target, uint64_t timeout_ns) {
  if (ld_acquire_u64(cnt) >= target) return true;
  return spin_geq_u64_slow(cnt, target, timeout_ns);
}

// Bounded spin until *cnt >= target. Returns false on timeout. The loop is out of line (one copy per kernel).
static __device__ __noinline__ bool spin_geq_slow(const uint32_t* cnt, uint32_t target, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 8; ++i) {
      if (ld_acquire_u32(cnt) >= target) return true;
      __nanosleep(20);
    }
    if (globaltimer() - t0 > timeout_ns) return false;
  }
}
__device__ __forceinline__ bool spin_geq(const uint32_t* cnt, uint32_t target, uint64_t timeout_ns) {
  if (ld_acquire_u32(cnt) >= target) return true;
  return spin_geq_slow(cnt, target, timeout_ns);
}

constexpr uint32_t MAGIC16 = 0x64006400u;   // fp16 pair (1024, 1024): codes OR-ed into the low mantissa bits

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
