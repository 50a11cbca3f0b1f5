#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.cuh"

namespace moe {

struct RepackSrc {   // canonical layout, device pointers
  const uint8_t *router_q; const uint16_t *router_s, *router_b;
  const uint8_t *exp_gate_q; const uint16_t *exp_gate_s, *exp_gate_b;
  const uint8_t *exp_up_q; const uint16_t *exp_up_s, *exp_up_b;
  const uint8_t *exp_down_q; const uint16_t *exp_down_s, *exp_down_b;
  const uint8_t *sh_gate_q; const uint16_t *sh_gate_s, *sh_gate_b;
  const uint8_t *sh_up_q; const uint16_t *sh_up_s, *sh_up_b;
  const uint8_t *sh_down_q; const uint16_t *sh_down_s, *sh_down_b;
};

struct RepackDst {
  uint8_t *router, *sh_gu, *sh_dn, *ex_gu, *ex_dn;
};

cudaError_t repack_all(const RepackSrc& w, const MoeLayout& L, const RepackDst& d, cudaStream_t st);
cudaError_t debug_dequant(const uint8_t* base, const MoeLayout& L, int which, int index, float* out,
                          cudaStream_t st);

}  // namespace moe
