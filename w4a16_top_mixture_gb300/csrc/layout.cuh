// Device-resident (repacked) layout of one block's weights, shared by the repack, debug and forward kernels.
//
// The canonical layout (see include/moe_block.h) is regrouped at load time so that every unit of work a CTA
// streams is one contiguous, 16-byte aligned range that a single bulk copy can move into shared memory:
//
//   router   [E+1][RR]     row r: int8 codes of the row, permuted (see moe_int8_perm), then H/64 (s,b) pairs
//   sh_gu    [Is][SU]      unit i: gate row codes (permuted) | up row codes (permuted) | gate (s,b) | up (s,b)
//   sh_dn    [H][SDR]      row r: Is int8 codes, 8-byte blocks in the in-block order below | Is/64 (s,b)
//   ex_gu    [E][I][EU]    unit (e,i): gate row int4 codes | up row int4 codes | gate (s,b) | up (s,b)
//   ex_dn    [E][H][DR]    row r of expert e's down matrix: I int4 codes | I/64 (s,b); a CTA's output rows of
//                          one expert are one contiguous range
//
// The code order inside a row serves the decode kernels' integer dot products, which take column pairs (0,1)
// (4,5) (2,3) (6,7) of every 8 columns: an int8 8-byte block holds columns 0 1 4 5 2 3 6 7; an int4 32-bit word
// holds columns 0..7 as bytes (c0|c2<<4, c1|c3<<4, c4|c6<<4, c5|c7<<4), so masking its low and high nibbles
// in place yields the same pairs. int8 rows of H columns (router, shared gate/up) are also interleaved in
// 16-byte blocks so that the lanes of a warp read consecutive 16 bytes: the 32-column chunk c = l + LW*p, half
// h (16 columns), lands at byte ((p*2 + h)*LW + l)*16 of the row, where LW = min(32, H/32) lanes work on a row.
#pragma once
#include <stddef.h>
#include <stdint.h>

#ifndef MOE_HD
#ifdef __CUDACC__
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif
#endif

MOE_HD size_t moe_align16(size_t v) { return (v + 15) & ~(size_t)15; }

struct MoeLayout {
  int H, E, K, I, Is;
  int GB, GI, GS;     // groups of 64 along H, I, Is
  int NCH, LW, P;     // 32-column chunks per H row, lanes per row, chunks per lane
  size_t RR, SU, SDR, EU, DR;
  size_t router_bytes, shgu_bytes, shdn_bytes, exgu_bytes, exdn_bytes;
  size_t exgu_expert, exdn_expert;
};

inline MoeLayout moe_make_layout(int H, int E, int K, int I, int Is) {
  MoeLayout L;
  L.H = H; L.E = E; L.K = K; L.I = I; L.Is = Is;
  L.GB = H / 64; L.GI = I / 64; L.GS = Is / 64;
  L.NCH = H / 32; L.LW = L.NCH < 32 ? L.NCH : 32; L.P = (L.NCH + 31) / 32;
  L.RR = moe_align16((size_t)H + (size_t)L.GB * 4);
  L.SU = moe_align16(2 * (size_t)H + 2 * (size_t)L.GB * 4);
  L.SDR = moe_align16((size_t)Is + (size_t)L.GS * 4);
  L.EU = moe_align16((size_t)H + 2 * (size_t)L.GB * 4);
  L.DR = moe_align16((size_t)I / 2 + (size_t)L.GI * 4);
  L.router_bytes = (size_t)(E + 1) * L.RR;
  L.shgu_bytes = (size_t)Is * L.SU;
  L.shdn_bytes = (size_t)H * L.SDR;
  L.exgu_expert = (size_t)I * L.EU;
  L.exdn_expert = (size_t)H * L.DR;
  L.exgu_bytes = (size_t)E * L.exgu_expert;
  L.exdn_bytes = (size_t)E * L.exdn_expert;
  return L;
}

// position of column k (0..7) inside an int8 8-byte block
MOE_HD int moe_int8_block_pos(int k) {
  const int pos8[8] = {0, 1, 4, 5, 2, 3, 6, 7};
  return pos8[k];
}
MOE_HD int moe_int8_block_col(int j) { return (j & ~7) + moe_int8_block_pos(j & 7); }

// bit position of column k (0..7) inside an int4 word of the decode layout
MOE_HD int moe_int4_shift(int k) {
  const int sh[8] = {0, 8, 4, 12, 16, 24, 20, 28};
  return sh[k];
}
// canonical word (column n at bits 4n) -> decode-layout word: columns 1 <-> 2 and 5 <-> 6 swap nibbles
MOE_HD uint32_t moe_int4_word(uint32_t w) {
  return (w & 0xF00FF00Fu) | ((w & 0x00F000F0u) << 4) | ((w & 0x0F000F00u) >> 4);
}

// byte position of int8 column j inside a permuted row. The 32-column chunk c = l + LW*p, half h (16
// columns), lands at ((p*2 + h)*LW + l)*16 so that the lanes of a warp read consecutive 16 bytes; inside each
// 8-byte block the columns are ordered 0 1 4 5 2 3 6 7, so that the byte pairs (0,2) and (1,3) of each 32-bit
// word hold the columns (k, 4+k) that the int4 rows also pair.
MOE_HD int moe_int8_perm(int j, int LW) {
  int c = j >> 5, within = j & 31, h = within >> 4, b = within & 15;
  int l = c % LW, p = c / LW;
  int blk = b >> 3, k = b & 7;
  return ((p * 2 + h) * LW + l) * 16 + blk * 8 + moe_int8_block_pos(k);
}
