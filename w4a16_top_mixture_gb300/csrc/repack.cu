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

// int8 rows: n_rows rows of `cols` codes -> permuted codes at dst + r*stride + base, (s,b) pairs after.
__global__ void k_repack_int8_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                   const uint16_t* __restrict__ b, uint8_t* __restrict__ dst, int n_rows,
                                   int cols, size_t stride, size_t code_off, size_t sb_off, int permute, int LW) {
  size_t n = (size_t)n_rows * cols;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    int r = (int)(i / cols), j = (int)(i % cols);
    int pos = permute ? moe_int8_perm(j, LW) : j;
    uint8_t* row = dst + (size_t)r * stride;
    row[code_off + pos] = q[i];
    if ((j & 63) == 0) {
      size_t g = (size_t)r * (cols / 64) + j / 64;
      *reinterpret_cast<uint32_t*>(row + sb_off + (j / 64) * 4) = sb_pair(s, b, g);
    }
  }
}

// int4 rows (packed bytes copied as they are): n_rows rows of cols/2 bytes.
__global__ void k_repack_int4_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                   const uint16_t* __restrict__ b, uint8_t* __restrict__ dst, int n_rows,
                                   int cols, size_t stride, size_t code_off, size_t sb_off) {
  size_t nb = (size_t)n_rows * (cols / 2);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nb; i += (size_t)gridDim.x * blockDim.x) {
    int r = (int)(i / (cols / 2)), jb = (int)(i % (cols / 2));
    uint8_t* row = dst + (size_t)r * stride;
    row[code_off + jb] = q[i];
    if ((jb & 31) == 0) {
      size_t g = (size_t)r * (cols / 64) + jb / 32;
      *reinterpret_cast<uint32_t*>(row + sb_off + (jb / 32) * 4) = sb_pair(s, b, g);
    }
  }
}

// ---------------------------------------------------------------- debug dequantisation
// which: 0 router, 1 expert gate, 2 expert up, 3 expert down, 4 shared gate, 5 shared up, 6 shared down.
// Output row-major in the canonical orientation. Every element goes through the forward kernels' unpack
// helpers and then w = fma(s, q, b) in fp32 (exactly the correctly rounded s*q + b).
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
    float v[8];
    if (which == 0 || which == 4 || which == 5) {
      const uint8_t* row;
      size_t sb_off;
      if (which == 0) { row = base + (size_t)r * L.RR; sb_off = L.H; }
      else { row = base + (size_t)r * L.SU + (which == 5 ? L.H : 0); sb_off = 2 * (size_t)L.H - (which == 5 ? L.H : 0) + (which == 5 ? (size_t)L.GB * 4 : 0); }
      // the 8-byte block of columns c8..c8+7 starts at the permuted position of column c8
      const uint8_t* blk = row + moe_int8_perm(c8, L.LW);
      uint32_t pr[4];
      int8_block_pairs(*reinterpret_cast<const uint32_t*>(blk), *reinterpret_cast<const uint32_t*>(blk + 4), pr);
      float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + sb_off + (c8 / 64) * 4));
      for (int k = 0; k < 4; ++k) {
        const float2 f = h2f(pr[k]);   // (1024 + c_k, 1024 + c_{4+k}) exactly
        v[k] = __fmaf_rn(sb.x, f.x - 1024.0f, sb.y);
        v[4 + k] = __fmaf_rn(sb.x, f.y - 1024.0f, sb.y);
      }
    } else if (which >= 1 && which <= 3) {
      // int4 rows: expert gate / up (units of gate row | up row | pairs) or down (row | pairs)
      const uint8_t* row;
      const uint8_t* sbp;
      if (which == 3) {
        row = base + ((size_t)index * L.H + r) * L.DR;
        sbp = row + L.I / 2;
      } else {
        const uint8_t* unit = base + ((size_t)index * L.I + r) * L.EU;
        row = unit + (which == 2 ? L.H / 2 : 0);
        sbp = unit + (size_t)L.H + (which == 2 ? (size_t)L.GB * 4 : 0);
      }
      uint32_t w = *reinterpret_cast<const uint32_t*>(row + c8 / 2);
      uint32_t pr[4];
      int4_word_pairs(w, pr);
      float2 sb = h2f(*reinterpret_cast<const uint32_t*>(sbp + (c8 / 64) * 4));
      for (int k = 0; k < 4; ++k) {
        const float2 f = h2f(pr[k]);   // 1024 + q (k even) or 1024 + 16 q (k odd), exactly
        const float sc = (k & 1) ? 0.0625f : 1.0f;
        v[k] = __fmaf_rn(sb.x, (f.x - 1024.0f) * sc, sb.y);
        v[4 + k] = __fmaf_rn(sb.x, (f.y - 1024.0f) * sc, sb.y);
      }
    } else {
      const uint8_t* row = base + (size_t)r * L.SDR;
      uint32_t w0 = *reinterpret_cast<const uint32_t*>(row + c8);
      uint32_t w1 = *reinterpret_cast<const uint32_t*>(row + c8 + 4);
      float2 q[4];
      unpack_int8_word(w0, q[0], q[1]);
      unpack_int8_word(w1, q[2], q[3]);
      float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + L.Is + (c8 / 64) * 4));
      for (int k = 0; k < 4; ++k) {
        v[2 * k] = __fmaf_rn(sb.x, q[k].x, sb.y);
        v[2 * k + 1] = __fmaf_rn(sb.x, q[k].y, sb.y);
      }
    }
    float* o = out + (size_t)r * cols + c8;
    for (int k = 0; k < 8; ++k) o[k] = v[k];
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
  // shared down rows (natural order)
  k_repack_int8_rows<<<grid_for((size_t)H * Is), 256, 0, st>>>(w.sh_down_q, w.sh_down_s, w.sh_down_b, d.sh_dn, H,
                                                                Is, L.SDR, 0, Is, 0, L.LW);
  // expert gate/up units: rows of all experts are consecutive (e*I + i)
  k_repack_int4_rows<<<grid_for((size_t)E * I * H / 2), 256, 0, st>>>(w.exp_gate_q, w.exp_gate_s, w.exp_gate_b,
                                                                       d.ex_gu, E * I, H, L.EU, 0, H);
  k_repack_int4_rows<<<grid_for((size_t)E * I * H / 2), 256, 0, st>>>(w.exp_up_q, w.exp_up_s, w.exp_up_b, d.ex_gu,
                                                                       E * I, H, L.EU, H / 2,
                                                                       (size_t)H + (size_t)L.GB * 4);
  // expert down rows: rows of all experts are consecutive (e*H + r)
  k_repack_int4_rows<<<grid_for((size_t)E * H * I / 2), 256, 0, st>>>(w.exp_down_q, w.exp_down_s, w.exp_down_b,
                                                                       d.ex_dn, E * H, I, L.DR, 0, I / 2);
  return cudaGetLastError();
}

cudaError_t debug_dequant(const uint8_t* base, const MoeLayout& L, int which, int index, float* out,
                          cudaStream_t st) {
  k_debug_dequant<<<1024, 256, 0, st>>>(base, L, which, index, out);
  return cudaGetLastError();
}

}  // namespace moe
