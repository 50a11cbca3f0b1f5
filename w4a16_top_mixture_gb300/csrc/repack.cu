// Load-time repacking of the canonical weights into the device layout of layout.cuh, and the debug export
// that dequantises a matrix back out of that layout with the same unpacking code the forward kernels use.
#include <cuda_fp16.h>
#include <stdint.h>

#include "layout.cuh"
#include "ptx.cuh"
#include "repack.cuh"

namespace moe {

__device__ __forceinline__ uint32_t sb_pair(const uint16_t* s, const uint16_t* b, size_t i) {
  return (uint32_t)s[i] | ((uint32_t)b[i] << 16);
}

// int8 rows: n_rows rows of `cols` codes -> codes at dst + r*stride + code_off, (s,b) pairs at sb_off. permute 1:
// lane-interleaved 16-byte halves of 32-column chunks with the in-block order (moe_int8_perm); 2: the in-block
// order only (columns 0 1 4 5 2 3 6 7 of every 8-byte block).
__global__ void k_repack_int8_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                   const uint16_t* __restrict__ b, uint8_t* __restrict__ dst, int n_rows,
                                   int cols, size_t stride, size_t code_off, size_t sb_off, int permute, int LW) {
  size_t n = (size_t)n_rows * cols;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    int r = (int)(i / cols), j = (int)(i % cols);
    int pos = permute == 1 ? moe_int8_perm(j, LW) : permute == 2 ? moe_int8_block_col(j) : j;
    uint8_t* row = dst + (size_t)r * stride;
    row[code_off + pos] = q[i];
    if ((j & 63) == 0) {
      size_t g = (size_t)r * (cols / 64) + j / 64;
      *reinterpret_cast<uint32_t*>(row + sb_off + (j / 64) * 4) = sb_pair(s, b, g);
    }
  }
}

// int4 rows: n_rows rows of cols/2 bytes, one 32-bit word (8 codes) per thread, re-laid from the canonical
// packing (code n at bits 4n) into the decode layout (moe_int4_word).
__global__ void k_repack_int4_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                   const uint16_t* __restrict__ b, uint8_t* __restrict__ dst, int n_rows,
                                   int cols, size_t stride, size_t code_off, size_t sb_off) {
  const int wpr = cols / 8;   // words per row
  size_t nw = (size_t)n_rows * wpr;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nw; i += (size_t)gridDim.x * blockDim.x) {
    int r = (int)(i / wpr), jw = (int)(i % wpr);
    uint8_t* row = dst + (size_t)r * stride;
    *reinterpret_cast<uint32_t*>(row + code_off + (size_t)jw * 4) = moe_int4_word(reinterpret_cast<const uint32_t*>(q)[i]);
    if ((jw & 7) == 0) {
      size_t g = (size_t)r * (cols / 64) + jw / 8;
      *reinterpret_cast<uint32_t*>(row + sb_off + (jw / 8) * 4) = sb_pair(s, b, g);
    }
  }
}

// ---------------------------------------------------------------- debug dequantisation
// which: 0 router, 1 expert gate, 2 expert up, 3 expert down, 4 shared gate, 5 shared up, 6 shared down.
// Output row-major in the canonical orientation. Each element's code is read back from its place in the decode
// layout (the positions the forward kernels' dot products pair with the activations) and dequantised as
// w = fma(s, q, b) in fp32, which is exactly the correctly rounded s*q + b.
__global__ void k_debug_dequant(const uint8_t* __restrict__ base, MoeLayout L, int which, int index,
                                float* __restrict__ out) {
  int rows, cols;
  switch (which) {
    case 0: rows = L.E + 1; cols = L.H; break;
    case 1: case 2: rows = L.I; cols = L.H; break;
    case 3: rows = L.H; cols = L.I; break;
    case 4: case 5: rows = L.Is; cols = L.H; break;
    default: rows = L.H; cols = L.Is; break;
  }
  // one thread per 8 consecutive columns of one row
  size_t n = (size_t)rows * (cols / 8);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    int r = (int)(i / (cols / 8));
    int c8 = (int)(i % (cols / 8)) * 8;
    int qv[8];
    const uint8_t* sbp;
    if (which == 0 || which == 4 || which == 5 || which == 6) {
      const uint8_t* row;
      const uint8_t* blk;
      if (which == 6) {
        row = base + (size_t)r * L.SDR;
        sbp = row + L.Is;
        blk = row + c8;                                       // in-block order only
      } else {
        if (which == 0) { row = base + (size_t)r * L.RR; sbp = row + L.H; }
        else {
          const uint8_t* unit = base + (size_t)r * L.SU;
          row = unit + (which == 5 ? L.H : 0);
          sbp = unit + 2 * (size_t)L.H + (which == 5 ? (size_t)L.GB * 4 : 0);
        }
        blk = row + moe_int8_perm(c8, L.LW);                  // the block of columns c8..c8+7
      }
      for (int k = 0; k < 8; ++k) qv[k] = blk[moe_int8_block_pos(k)];
    } else {
      // int4 rows: expert gate / up (units of gate row | up row | pairs) or down (row | pairs)
      const uint8_t* row;
      if (which == 3) {
        row = base + ((size_t)index * L.H + r) * L.DR;
        sbp = row + L.I / 2;
      } else {
        const uint8_t* unit = base + ((size_t)index * L.I + r) * L.EU;
        row = unit + (which == 2 ? L.H / 2 : 0);
        sbp = unit + (size_t)L.H + (which == 2 ? (size_t)L.GB * 4 : 0);
      }
      const uint32_t w = *reinterpret_cast<const uint32_t*>(row + c8 / 2);
      for (int k = 0; k < 8; ++k) qv[k] = (int)((w >> moe_int4_shift(k)) & 0xFu);
    }
    const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(sbp + (c8 / 64) * 4));
    float* o = out + (size_t)r * cols + c8;
    for (int k = 0; k < 8; ++k) o[k] = __fmaf_rn(sb.x, (float)qv[k], sb.y);
  }
}

static int grid_for(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 65535 * 8) g = 65535 * 8;
  if (g < 1) g = 1;
  return (int)g;
}

cudaError_t repack_all(const RepackSrc& w, const MoeLayout& L, const RepackDst& d, cudaStream_t st) {
  const int H = L.H, E = L.E, I = L.I, Is = L.Is;
  // router: E+1 int8 rows, permuted
  k_repack_int8_rows<<<grid_for((size_t)(E + 1) * H), 256, 0, st>>>(w.router_q, w.router_s, w.router_b, d.router,
                                                                     E + 1, H, L.RR, 0, H, 1, L.LW);
  // shared gate/up units
  k_repack_int8_rows<<<grid_for((size_t)Is * H), 256, 0, st>>>(w.sh_gate_q, w.sh_gate_s, w.sh_gate_b, d.sh_gu, Is,
                                                                H, L.SU, 0, 2 * (size_t)H, 1, L.LW);
  k_repack_int8_rows<<<grid_for((size_t)Is * H), 256, 0, st>>>(w.sh_up_q, w.sh_up_s, w.sh_up_b, d.sh_gu, Is, H,
                                                                L.SU, H, 2 * (size_t)H + (size_t)L.GB * 4, 1, L.LW);
  // shared down rows (in-block order)
  k_repack_int8_rows<<<grid_for((size_t)H * Is), 256, 0, st>>>(w.sh_down_q, w.sh_down_s, w.sh_down_b, d.sh_dn, H,
                                                                Is, L.SDR, 0, Is, 2, L.LW);
  // expert gate/up units: rows of all experts are consecutive (e*I + i)
  k_repack_int4_rows<<<grid_for((size_t)E * I * H / 8), 256, 0, st>>>(w.exp_gate_q, w.exp_gate_s, w.exp_gate_b,
                                                                       d.ex_gu, E * I, H, L.EU, 0, H);
  k_repack_int4_rows<<<grid_for((size_t)E * I * H / 8), 256, 0, st>>>(w.exp_up_q, w.exp_up_s, w.exp_up_b, d.ex_gu,
                                                                       E * I, H, L.EU, H / 2,
                                                                       (size_t)H + (size_t)L.GB * 4);
  // expert down rows: rows of all experts are consecutive (e*H + r)
  k_repack_int4_rows<<<grid_for((size_t)E * H * I / 8), 256, 0, st>>>(w.exp_down_q, w.exp_down_s, w.exp_down_b,
                                                                       d.ex_dn, E * H, I, L.DR, 0, I / 2);
  return cudaGetLastError();
}

cudaError_t debug_dequant(const uint8_t* base, const MoeLayout& L, int which, int index, float* out,
                          cudaStream_t st) {
  k_debug_dequant<<<1024, 256, 0, st>>>(base, L, which, index, out);
  return cudaGetLastError();
}

}  // namespace moe
