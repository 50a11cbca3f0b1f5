#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.cuh"

namespace moe {

constexpr int DEC_NCW = 16;                       // consumer warps
constexpr int DEC_THREADS = (DEC_NCW + 1) * 32;   // + one producer warp
constexpr int DEC_TMAX = 16;                      // largest T of the fused decode kernel
constexpr int DEC_MAXSEG = 4;                     // expert segments one CTA's unit range may touch
constexpr int DEC_MAXROWS = 32;                   // output rows one CTA owns (ceil(H / grid))
constexpr int DEC_MAXNS = 24;                     // ring stages
constexpr int DEC_MAXGRID = 160;                  // CTAs (one per SM)
constexpr int DEC1_NCW = 12;                      // consumer warps of the single-token kernel
constexpr int DEC1_THREADS = (DEC1_NCW + 1) * 32; // + one producer warp

// device error bits
enum : uint32_t {
  ERR_WAIT_LOGITS = 1u, ERR_WAIT_HS = 2u, ERR_WAIT_H = 4u, ERR_WAIT_FULL = 8u, ERR_WAIT_EMPTY = 16u,
  ERR_WAIT_ROUTE = 32u, ERR_SEGMENTS = 64u,
  ERR_REFUSED = 128u,   // the single-token kernel found an earlier error not yet cleared and computed nothing
};

// Words of the handle's counter array (uint32 units). The multi-token kernel's counts (reset by its last CTA),
// the status word, and the single-token kernel's epoch and its two 64-bit exchange counts, which only grow:
// launch ep waits for ep * Is shared units and ep * K * I routed units.
constexpr int CNT_STATUS = 4, CNT_EPOCH = 5, CNT_HS64 = 8, CNT_H64 = 10, CNT_WORDS = 16;

// copies of the single-token kernel's published router logits (each CTA polls one), 256-byte aligned apart
#ifndef MOE_XLOG_COPIES
#define MOE_XLOG_COPIES 16
#endif
constexpr int XLOG_COPIES = MOE_XLOG_COPIES;
__host__ __device__ constexpr size_t xlog_stride(int E) { return (size_t)((E + 1 + 31) & ~31); }

struct DecodeArgs {
  const uint8_t *router, *sh_gu, *sh_dn, *ex_gu, *ex_dn;
  const uint16_t* x;        // [T][H] fp16 (h_in in residual mode)
  uint16_t* out;            // [T][H] fp16
  uint16_t* out2;           // optional second copy of out (a stacked layer's per-layer record); may be null
  const uint16_t* gamma;    // non-null: residual mode, x_hat = RMSNorm(x), out = x + block(x_hat)
  float eps;
  int T;
  float* logits;            // [T][E+1] (the single-token kernel writes it only as CTA 0's record)
  uint64_t* xlog;           // [XLOG_COPIES][xlog_stride(E)] the single-token kernel's router logits, published
                            // as {logit, epoch} words, every copy alike
  float* hs;                // [T][Is]
  float* hbuf;              // [T*K][I] routed h, one row per (expert, token) pair in expert-sorted order
  uint32_t* counters;       // [CNT_WORDS], see CNT_*
  uint32_t* status;
  int32_t* rec_ids;         // routing record [T][K] (written by CTA 0)
  float* rec_w;             // [T][K]
  float* rec_sg;            // [T]
  uint64_t timeout_ns;
  int skip_arrive;
  uint64_t* trace;          // optional [grid][32] globaltimer stamps at phase boundaries (debug)
};

struct DecodeLaunch {
  int grid, smem, NS, SS, hp;   // hp: routed h vectors staged in shared memory (one token: K; else 0)
};

// Launch plan of the single-token kernel: grid, dynamic shared memory, and whether two CTAs fit on one SM
// (so that the next call's CTAs can be resident while this call runs).
struct Decode1Launch {
  int grid, smem, two_per_sm;
};

// Host: shared-memory plan for a call with T tokens; returns false if it does not fit.
bool decode_plan(const MoeLayout& L, int T, int grid, int max_smem, DecodeLaunch* out);
bool decode_supported(const MoeLayout& L);   // shapes with a compiled decode kernel
cudaError_t decode_launch(const MoeLayout& L, const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st);
size_t decode_hbuf_floats(const MoeLayout& L, int T);

// Host: plan of the single-token kernel (T = 1); false if the shape has no such kernel or it does not fit.
bool decode1_plan(const MoeLayout& L, int grid, int max_smem, Decode1Launch* out);
cudaError_t decode1_launch(const MoeLayout& L, const DecodeArgs& a, const Decode1Launch& pl, cudaStream_t st);

// Host, on the current device: give the kernel of a plan its shared-memory limits and report how many of its
// CTAs one SM holds at once (the grid-wide counts of both decode kernels need the whole grid resident).
cudaError_t decode1_occupancy(const MoeLayout& L, const Decode1Launch& pl, int* ctas_per_sm);
cudaError_t decode_occupancy(const MoeLayout& L, const DecodeLaunch& pl, int* ctas_per_sm);

}  // namespace moe
