// Prompt-chunk path (T > 16 tokens): grouped GEMMs on the tcgen05 tensor cores.
//
// Weights for this path live in a second, GEMM-friendly copy ("GEMM layout"), built at load time for handles
// whose max_tokens exceeds the decode kernel's limit. Every matrix (rows = output units, columns = the
// reduction dimension) is cut into 128-row x 64-column tiles, one quantisation group wide; the tiles of a
// 128-row band are stored one after the other, and one tile is a single contiguous block:
//   codes  128 rows x 64 codes   int4: 32 bytes a row (canonical packing), int8: 64 bytes a row (P8 bytes)
//   pairs  128 (s, b) fp16 pairs, one 32-bit word a row
// so a K-tile of a band is one bulk copy (4608 bytes int4, 8704 bytes int8). Matrices:
//   router       int8  Mr x H    rows 0..E (E+1..Mr-1 zero), Mr = E+1 rounded up to 128
//   shared g/u   int8  2Is x H   band m = gate units 64m..64m+63, then the matching up units
//   shared down  int8  H x Is
//   expert g/u   int4  E x 2I x H, banded like the shared gate/up
//   expert down  int4  E x H x I
// Int8 rows have the bytes of each 8-byte block in the order 0 1 4 5 2 3 6 7 so that int8 and int4 rows both
// yield the column pairs (k, 4+k) of an 8-column block; activations are stored in the matching order
// (0 4 1 5 2 6 3 7 per 8 columns, "P8"), which leaves every dot product unchanged.
//
// The GEMM (chunk_gemm.cu) forms each K-tile's scaled codes s * q as an exact pair of fp16 halves A1 + A2 in
// tensor memory and accumulates A1 x + A2 x for a whole job in one fp32 accumulator; the offset term
// sum_g b_g sum(x over group g) is one more MMA per job against the activation rows' group sums. The group sums
// are made once per activation row by the kernel that writes the row (the prologue, the gather, the SwiGLU
// epilogue), as one 128-byte row of fp16 hi + lo pairs. Activation tiles and group-sum rows arrive by TMA tensor
// loads (128-byte swizzled, the layout the MMA reads) through tensor maps made once per handle.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.cuh"
#include "repack.cuh"

namespace moe {

constexpr int GEMM_BLK4 = 128 * 32 + 128 * 4;   // bytes of an int4 tile
constexpr int GEMM_BLK8 = 128 * 64 + 128 * 4;   // bytes of an int8 tile

struct GemmLayout {
  int H, E, K, I, Is, Mr;
  uint8_t *gr, *gsgu, *gsdn, *gegu, *gedn;   // tile blocks, band-major then K-tile
  size_t gegu_expert, gedn_expert;           // bytes per expert
};

// byte size of the GEMM-layout store for a block shape
size_t gemm_store_bytes(const MoeLayout& L);
// carve a GEMM layout out of `base` (gemm_store_bytes bytes, 256-byte aligned)
GemmLayout gemm_layout_carve(const MoeLayout& L, uint8_t* base);
// repack into the GEMM layout; *range_bad (a device word) ends up nonzero when a scale is out of the GEMM's range
// (see k_gemm_tiles)
cudaError_t gemm_repack(const RepackSrc& w, const GemmLayout& G, uint32_t* range_bad, cudaStream_t st);

constexpr int CHUNK_NT = 64;   // tokens (rows of activations) per GEMM tile
// The router's GEMM is split along K into up to ROUTER_SPLIT parts of a multiple of 8 K-tiles each (the offset
// term's MMA takes 8 groups per K step), each part a job of its own writing partial logits; the routing adds
// the parts in order.
constexpr int ROUTER_SPLIT = 4;
__host__ __device__ constexpr int router_kpp(int kt) { return (((kt + ROUTER_SPLIT - 1) / ROUTER_SPLIT) + 7) & ~7; }
__host__ __device__ constexpr int router_parts(int kt) { return (kt + router_kpp(kt) - 1) / router_kpp(kt); }
// row stride (floats) of the partial logits: E + 1 rounded up to 4, so that a lane reads its logits as float4s
__host__ __device__ constexpr int logit_stride(int e) { return (e + 1 + 3) & ~3; }

// scratch of the chunk path for up to Tm tokens. The group sums of an activation row (the sum of each
// 64-column group, in fp32) are stored as one 128-byte row of fp16 per activation row: element 2g holds the sum
// of group g rounded to fp16, element 2g + 1 the remainder rounded to fp16 (hi + lo carries ~22 bits), the rest
// zero. The GEMM loads a job's rows of them with one TMA tensor load, the B operand of the job's offset term.
constexpr int GSUM_COLS = 64;   // fp16 per group-sum row: at most 32 groups
struct ChunkScratch {
  uint16_t* xp;        // [Tm][H] fp16, P8 order (block input, after RMSNorm in residual mode)
  float* logits;       // [parts][T][logit_stride(E)] partial router logits (parts = router_parts(H / 64))
  uint16_t* hs;        // [Tm][Is] fp16, P8 order: RN_fp16(h) of the shared expert
  uint16_t* hs_lo;     // [Tm][Is] fp16, P8 order: RN_fp16(4096 (h - hs)), the low half of the split
  float* ys;           // [Tm][H] shared-expert output
  int32_t* ids;        // [Tm][K]
  float* w;            // [Tm][K]
  float* sg;           // [Tm]
  uint32_t* masks;     // [E][Tm/32] tokens routed to each expert
  int32_t* slot_of;    // [Tm][K] row of (token, j) in the expert-sorted order
  int32_t* tok_of;     // [Tm*K] token of each sorted row
  uint16_t* xs;        // [Tm*K][H] fp16 P8, activations gathered in sorted order
  uint16_t* hh;        // [Tm*K][I] fp16 P8, routed h (high half)
  uint16_t* hh_lo;     // [Tm*K][I] fp16 P8, routed h (low half, scaled by 4096)
  float* y;            // [Tm*K][H] routed expert outputs (unweighted)
  int4* groups;        // [E + Tm*K/CHUNK_NT + 1] (expert, first sorted row, rows) per row tile
  int32_t* ctl;        // [16] ctl[0] row-tile count, ctl[1] rows of the widest row tile; ctl[8] the weight
                       // repack's scale-range flag
  uint16_t* gs_xp;     // [Tm][64]   group sums of xp's rows
  uint16_t* gs_xs;     // [Tm*K][64] group sums of xs's rows
  uint16_t* gs_hs;     // [Tm][64]   group sums of hs + hs_lo / 4096
  uint16_t* gs_hh;     // [Tm*K][64] group sums of hh + hh_lo / 4096
};
size_t chunk_scratch_bytes(const MoeLayout& L, int Tm);
ChunkScratch chunk_scratch_carve(const MoeLayout& L, int Tm, uint8_t* base);

// TMA tensor maps of the GEMMs' activation operands: [buffer][box], boxes of 64 columns x 16, 32 or 64 rows,
// 128-byte swizzle, rows past the buffer read as zero
enum : int { CM_XP = 0, CM_XS, CM_HS, CM_HSLO, CM_HH, CM_HHLO, CM_GXP, CM_GXS, CM_GHS, CM_GHH, CM_COUNT };
constexpr int CM_BOXES = 3;
struct ChunkMaps {
  CUtensorMap m[CM_COUNT][CM_BOXES];
};
cudaError_t chunk_make_maps(const MoeLayout& L, const ChunkScratch& S, int Tm, ChunkMaps* out);

// GEMM launch of one phase: 1 router (in K parts), 2 expert + shared gate/up, 3 expert down + shared down
struct GemmArgs {
  GemmLayout G;
  ChunkScratch S;
  int T;             // tokens
  int Tm;            // row capacity of the per-token arrays (sum strides)
  int phase;
  uint32_t* status;
  uint64_t timeout_ns;
  uint64_t* trace;   // optional: CTA 0's SM-clock stamps of its first 64 K-tiles, [role event][64]
  ChunkMaps maps;
  int skip;          // test hook: CTA 0 withholds its first K-tile's copies, so its bounded waits run out
};
cudaError_t chunk_gemm_launch(const GemmArgs& g, int grid, cudaStream_t st);

// out[T][H] = block(x) (or h + block(RMSNorm(h)) when gamma != NULL) for T tokens, T <= Tm
cudaError_t chunk_forward(const MoeLayout& L, const GemmLayout& G, const ChunkScratch& S, const ChunkMaps& maps,
                          int Tm, int num_sms,
                          const uint16_t* x, uint16_t* out, int T, const uint16_t* gamma, float eps,
                          int32_t* rec_ids, float* rec_w, float* rec_sg, uint32_t* status, uint64_t timeout_ns,
                          uint64_t* trace, cudaStream_t st, int* launches, int skip = 0);

}  // namespace moe
