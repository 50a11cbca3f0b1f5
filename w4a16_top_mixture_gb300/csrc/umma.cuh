// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory allocation, shared-memory matrix
// descriptors for K-major operands in the 128-byte swizzled layout, the kind::f16 instruction descriptor, the
// MMA issue / commit, and tensor-memory loads for the epilogue.
//
// Operand layout used throughout (K-major, 128B swizzle): a tile of R rows x 64 fp16 (128 bytes per row) is
// stored row after row; inside each row the 16-byte chunk c (8 elements) sits at chunk position c ^ (row % 8);
// groups of 8 rows (1024 bytes) follow each other. Tile bases are 1024-byte aligned. One MMA consumes K = 16
// (32 bytes of each row); the next K step starts 32 bytes further into the rows.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace moe {

// byte offset of element chunk c (0..7) of row r in a K-major 128B-swizzled tile of 64-element rows
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

// shared-memory matrix descriptor: start address, leading byte offset (unused for swizzled K-major), stride
// byte offset 1024 (between 8-row groups), descriptor version 1, swizzle mode 2 (128B)
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor of kind::f16: fp16 A and B, fp32 accumulator, both K-major, M x N
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (0u << 7) | (0u << 10)           // A, B format: f16
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one M x N x 16 step; accumulate = 0 overwrites D
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, one M x N x 16 step. A occupies 8 consecutive columns from a_tmem: lane i
// holds row i, column c holds the fp16 pair (K = 2c, 2c + 1) in its low and high halves.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The MMAs of one K-tile (64 columns) as one issue sequence: for each 16-column K step k, D += A[k] B[k] then
// D += A[32 + k] B[k], A at TMEM columns a + 8k and a + 32 + 8k, B at descriptor b + 2k (its start address
// advanced by 32 bytes). The descriptor is passed as its two halves (the start address sits in the low half and
// never carries into the high one), so the steps need 32-bit adds only; the first MMA accumulates onto D only
// if acc_first is nonzero. PAIRS = false: the single sequence D += A[k] B[k] (A columns a + 8k).
template <bool PAIRS>
__device__ __forceinline__ void umma_f16_ktile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                               uint32_t idesc, uint32_t acc_first) {
  if (PAIRS) {
    asm volatile(
        "{\n .reg .pred pf, pt;\n .reg .b32 l1, l2, l3, x1, x2, x3, y0, y1, y2, y3;\n .reg .b64 q0, q1, q2, q3;\n"
        " setp.ne.b32 pf, %5, 0;\n setp.eq.b32 pt, %4, %4;\n"
        " add.u32 l1, %2, 2;\n add.u32 l2, %2, 4;\n add.u32 l3, %2, 6;\n"
        " mov.b64 q0, {%2, %3};\n mov.b64 q1, {l1, %3};\n mov.b64 q2, {l2, %3};\n mov.b64 q3, {l3, %3};\n"
        " add.u32 x1, %1, 8;\n add.u32 x2, %1, 16;\n add.u32 x3, %1, 24;\n"
        " add.u32 y0, %1, 32;\n add.u32 y1, %1, 40;\n add.u32 y2, %1, 48;\n add.u32 y3, %1, 56;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], q0, %4, pf;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [y0], q0, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], q1, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [y1], q1, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], q2, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [y2], q2, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], q3, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [y3], q3, %4, pt;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc_first)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred pf, pt;\n .reg .b32 l1, l2, l3, x1, x2, x3;\n .reg .b64 q0, q1, q2, q3;\n"
        " setp.ne.b32 pf, %5, 0;\n setp.eq.b32 pt, %4, %4;\n"
        " add.u32 l1, %2, 2;\n add.u32 l2, %2, 4;\n add.u32 l3, %2, 6;\n"
        " mov.b64 q0, {%2, %3};\n mov.b64 q1, {l1, %3};\n mov.b64 q2, {l2, %3};\n mov.b64 q3, {l3, %3};\n"
        " add.u32 x1, %1, 8;\n add.u32 x2, %1, 16;\n add.u32 x3, %1, 24;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], q0, %4, pf;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], q1, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], q2, %4, pt;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], q3, %4, pt;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc_first)
        : "memory");
  }
}
// mbarrier arrives once all previously issued MMAs of this thread have completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive columns: thread (lane) i receives row (lane base + i), columns col..col+15, in r.
// tcgen05.ld fills its destination registers asynchronously: they hold the loaded values only once
// tcgen05.wait::ld has returned. The compiler knows nothing of that, so the wait must name the registers as
// read and written (tmem_wait_ld below): otherwise it may schedule register-only uses of them (a conversion, an
// FMA) ahead of the wait, and those would read whatever the registers held before.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// waits for this thread's earlier tcgen05.ld operations; r: the destination registers of one of them, which
// are valid from here on (call it once per load whose registers are used; the waits after the first return
// at once)
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// 32 lanes x 32 consecutive columns: thread (lane) i writes row (lane base + i), columns col..col+31; returns
// once the stores have completed
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive columns, without the wait: issue several stores, then one tmem_wait_st()
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 1 column, without the wait
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 4-byte asynchronous global -> shared copy through L1 (zero-filled when src_bytes == 0)
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
// the mbarrier receives one arrival once every cp.async this thread issued so far has landed (the arrival is
// counted in the barrier's expected count: no increment)
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16-byte asynchronous global -> shared copy (zero-filled when src_bytes == 0)
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace moe
