// Prompt-chunk path (T > 16 tokens): grouped GEMMs on the tcgen05 tensor cores.
//
// Weights for this path live in a second, GEMM-friendly copy ("GEMM layout"), built at load time for handles
// whose max_tokens exceeds the decode kernel's limit:
//   gr    router      int8 [Mr][H]  rows 0..E (E+1..Mr-1 zero), Mr = E+1 rounded up to 128
//   gsgu  shared g/u  int8 [2Is][H] rows tile-interleaved: 128-row tile m = gate units 64m..64m+63, then up units
//   gsdn  shared down int8 [H][Is]
//   gegu  expert g/u  int4 [E][2I][H/2] tile-interleaved like gsgu, codes two per byte (canonical packing)
//   gedn  expert down int4 [E][H][I/2]
// Every int8 row has its bytes permuted inside each 8-byte block as columns 0 1 4 5 2 3 6 7, so that int8 and
// int4 rows both yield the column pairs (k, 4+k) of an 8-column block; activations are stored in the matching
// order (0 4 1 5 2 6 3 7 per 8 columns, "P8"), which leaves every dot product unchanged. The (s, b) pairs of each
// matrix are stored group-major: sb[g][row] (one 32-bit fp16 pair), so a K-tile of 128 rows is one 512-byte run.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.cuh"
#include "repack.cuh"

namespace moe {

struct GemmLayout {
  int H, E, K, I, Is, Mr;
  uint8_t *gr, *gsgu, *gsdn, *gegu, *gedn;       // codes
  uint32_t *grs, *gsgus, *gsdns, *gegus, *gedns;  // (s, b) pairs, group-major
  size_t gegu_expert, gedn_expert, gegus_expert, gedns_expert;   // per-expert strides (bytes / pairs)
};

// byte sizes of the GEMM-layout store (codes + pairs) for a block shape
size_t gemm_store_bytes(const MoeLayout& L);
// carve a GEMM layout out of `base` (gemm_store_bytes bytes, 256-byte aligned)
GemmLayout gemm_layout_carve(const MoeLayout& L, uint8_t* base);
cudaError_t gemm_repack(const RepackSrc& w, const GemmLayout& G, cudaStream_t st);

// scratch of the chunk path for up to Tm tokens
struct ChunkScratch {
  uint16_t* xp;        // [Tm][H] fp16, P8 order (block input, after RMSNorm in residual mode)
  float* logits;       // [Tm][E+1]
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
  int4* groups;        // [E + Tm*K/256 + 1] (expert, first sorted row, rows) per 256-row tile group
  int32_t* ctl;        // [16] counters: job counters, group count
};
size_t chunk_scratch_bytes(const MoeLayout& L, int Tm);
ChunkScratch chunk_scratch_carve(const MoeLayout& L, int Tm, uint8_t* base);

// out[T][H] = block(x) (or h + block(RMSNorm(h)) when gamma != NULL) for T tokens, T <= Tm
cudaError_t chunk_forward(const MoeLayout& L, const GemmLayout& G, const ChunkScratch& S, int num_sms,
                          const uint16_t* x, uint16_t* out, int T, const uint16_t* gamma, float eps,
                          int32_t* rec_ids, float* rec_w, float* rec_sg, uint32_t* status, uint64_t timeout_ns,
                          cudaStream_t st, int* launches);

}  // namespace moe
