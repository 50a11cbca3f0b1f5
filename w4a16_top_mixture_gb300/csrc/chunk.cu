// Prompt-chunk path of the W4A16 routed-MoE block (T > 16): weight repack into the GEMM layout, the tcgen05
// grouped-GEMM kernel, routing / bucketing / gather kernels and the final combine. See chunk.cuh.
#include <cuda_fp16.h>
#include <stdint.h>

#include "chunk.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace moe {

static size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t gemm_store_bytes(const MoeLayout& L) {
  const size_t H = L.H, E = L.E, I = L.I, Is = L.Is, Mr = ((L.E + 1 + 127) / 128) * 128;
  size_t b = 0;
  b += al256(Mr * H) + al256((H / 64) * Mr * 4);                 // router
  b += al256(2 * Is * H) + al256((H / 64) * 2 * Is * 4);         // shared gate/up
  b += al256(H * Is) + al256((Is / 64) * H * 4);                 // shared down
  b += al256(E * 2 * I * (H / 2)) + al256(E * (H / 64) * 2 * I * 4);   // expert gate/up
  b += al256(E * H * (I / 2)) + al256(E * (I / 64) * H * 4);           // expert down
  return b;
}

GemmLayout gemm_layout_carve(const MoeLayout& L, uint8_t* base) {
  GemmLayout G;
  G.H = L.H; G.E = L.E; G.K = L.K; G.I = L.I; G.Is = L.Is;
  G.Mr = ((L.E + 1 + 127) / 128) * 128;
  const size_t H = L.H, E = L.E, I = L.I, Is = L.Is, Mr = G.Mr;
  uint8_t* p = base;
  auto take = [&](size_t n) { uint8_t* r = p; p += al256(n); return r; };
  G.gr = take(Mr * H);
  G.grs = (uint32_t*)take((H / 64) * Mr * 4);
  G.gsgu = take(2 * Is * H);
  G.gsgus = (uint32_t*)take((H / 64) * 2 * Is * 4);
  G.gsdn = take(H * Is);
  G.gsdns = (uint32_t*)take((Is / 64) * H * 4);
  G.gegu = take(E * 2 * I * (H / 2));
  G.gegus = (uint32_t*)take(E * (H / 64) * 2 * I * 4);
  G.gedn = take(E * H * (I / 2));
  G.gedns = (uint32_t*)take(E * (I / 64) * H * 4);
  G.gegu_expert = 2 * I * (H / 2);
  G.gedn_expert = H * (I / 2);
  G.gegus_expert = (H / 64) * 2 * I;
  G.gedns_expert = (I / 64) * H;
  return G;
}

// One thread per (batch, row, 8-byte block of codes): copies a quantised row into the GEMM layout. rowmode 0
// keeps the row index; 1 / 2 place row r of a gate / up matrix into its 128-row tile (r/64)*128 + (0 | 64) +
// r%64. perm8 reorders the bytes of each 8-byte block as 0 1 4 5 2 3 6 7 (int8 rows). The (s, b) pair of each
// (row, group) goes to dsb[group][drow].
__global__ void k_gemm_rows(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                            const uint16_t* __restrict__ b, int nbatch, int nrows, int rowbytes, int groups,
                            size_t src_q_batch, size_t src_sb_batch, uint8_t* __restrict__ dq,
                            uint32_t* __restrict__ dsb, int drows, size_t dst_q_batch, size_t dst_sb_batch,
                            int rowmode, int perm8) {
  const int blocks = rowbytes / 8;
  const size_t n = (size_t)nbatch * nrows * blocks;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int blk = (int)(i % blocks);
    const size_t t = i / blocks;
    const int r = (int)(t % nrows);
    const int bt = (int)(t / nrows);
    const int dr = rowmode == 0 ? r : (r / 64) * 128 + (rowmode == 2 ? 64 : 0) + r % 64;
    const uint8_t* src = q + bt * src_q_batch + (size_t)r * rowbytes + blk * 8;
    uint8_t* dst = dq + bt * dst_q_batch + (size_t)dr * rowbytes + blk * 8;
    if (perm8) {
      const int pos[8] = {0, 1, 4, 5, 2, 3, 6, 7};   // dst byte j holds column pos[j]
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = src[pos[j]];
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = src[j];
    }
    // one thread per (row, group) writes the pair: the first block of each 64-column group
    const int cols_per_blk = perm8 ? 8 : 16;
    const int col0 = blk * cols_per_blk;
    if (col0 % 64 == 0) {
      const int g = col0 / 64;
      const size_t si = bt * src_sb_batch + (size_t)r * groups + g;
      dsb[bt * dst_sb_batch + (size_t)g * drows + dr] = (uint32_t)s[si] | ((uint32_t)b[si] << 16);
    }
  }
}

static int grid_for_n(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 65535 * 8) g = 65535 * 8;
  return g < 1 ? 1 : (int)g;
}

cudaError_t gemm_repack(const RepackSrc& w, const GemmLayout& G, cudaStream_t st) {
  const int H = G.H, E = G.E, I = G.I, Is = G.Is;
  cudaError_t e = cudaMemsetAsync(G.gr, 0, (size_t)G.Mr * H, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(G.grs, 0, (size_t)(H / 64) * G.Mr * 4, st);
  if (e != cudaSuccess) return e;
  auto rows = [&](const uint8_t* q, const uint16_t* s, const uint16_t* b, int nbatch, int nrows, int rowbytes,
                  int groups, size_t sqb, size_t ssb, uint8_t* dq, uint32_t* dsb, int drows, size_t dqb,
                  size_t dsbb, int rowmode, int perm8) {
    const size_t n = (size_t)nbatch * nrows * (rowbytes / 8);
    k_gemm_rows<<<grid_for_n(n), 256, 0, st>>>(q, s, b, nbatch, nrows, rowbytes, groups, sqb, ssb, dq, dsb, drows,
                                               dqb, dsbb, rowmode, perm8);
  };
  rows(w.router_q, w.router_s, w.router_b, 1, E + 1, H, H / 64, 0, 0, G.gr, G.grs, G.Mr, 0, 0, 0, 1);
  rows(w.sh_gate_q, w.sh_gate_s, w.sh_gate_b, 1, Is, H, H / 64, 0, 0, G.gsgu, G.gsgus, 2 * Is, 0, 0, 1, 1);
  rows(w.sh_up_q, w.sh_up_s, w.sh_up_b, 1, Is, H, H / 64, 0, 0, G.gsgu, G.gsgus, 2 * Is, 0, 0, 2, 1);
  rows(w.sh_down_q, w.sh_down_s, w.sh_down_b, 1, H, Is, Is / 64, 0, 0, G.gsdn, G.gsdns, H, 0, 0, 0, 1);
  rows(w.exp_gate_q, w.exp_gate_s, w.exp_gate_b, E, I, H / 2, H / 64, (size_t)I * (H / 2), (size_t)I * (H / 64),
       G.gegu, G.gegus, 2 * I, G.gegu_expert, G.gegus_expert, 1, 0);
  rows(w.exp_up_q, w.exp_up_s, w.exp_up_b, E, I, H / 2, H / 64, (size_t)I * (H / 2), (size_t)I * (H / 64), G.gegu,
       G.gegus, 2 * I, G.gegu_expert, G.gegus_expert, 2, 0);
  rows(w.exp_down_q, w.exp_down_s, w.exp_down_b, E, H, I / 2, I / 64, (size_t)H * (I / 2), (size_t)H * (I / 64),
       G.gedn, G.gedns, H, G.gedn_expert, G.gedns_expert, 0, 0);
  return cudaGetLastError();
}

size_t chunk_scratch_bytes(const MoeLayout& L, int Tm) {
  const size_t H = L.H, E = L.E, K = L.K, I = L.I, Is = L.Is, T = Tm, TK = (size_t)Tm * L.K;
  const size_t TW = (T + 31) / 32;
  size_t b = 0;
  b += al256(T * H * 2) + al256(T * (E + 1) * 4) + al256(T * Is * 2) * 2 + al256(T * H * 4);
  b += al256(T * K * 4) * 2 + al256(T * 4) + al256(E * TW * 4) + al256(T * K * 4) + al256(TK * 4);
  b += al256(TK * H * 2) + al256(TK * I * 2) * 2 + al256(TK * H * 4);
  b += al256((E + TK / 256 + 2) * 16) + al256(16 * 4);
  return b;
}

ChunkScratch chunk_scratch_carve(const MoeLayout& L, int Tm, uint8_t* base) {
  const size_t H = L.H, E = L.E, K = L.K, I = L.I, Is = L.Is, T = Tm, TK = (size_t)Tm * L.K;
  const size_t TW = (T + 31) / 32;
  uint8_t* p = base;
  auto take = [&](size_t n) { uint8_t* r = p; p += al256(n); return r; };
  ChunkScratch S;
  S.xp = (uint16_t*)take(T * H * 2);
  S.logits = (float*)take(T * (E + 1) * 4);
  S.hs = (uint16_t*)take(T * Is * 2);
  S.hs_lo = (uint16_t*)take(T * Is * 2);
  S.ys = (float*)take(T * H * 4);
  S.ids = (int32_t*)take(T * K * 4);
  S.w = (float*)take(T * K * 4);
  S.sg = (float*)take(T * 4);
  S.masks = (uint32_t*)take(E * TW * 4);
  S.slot_of = (int32_t*)take(T * K * 4);
  S.tok_of = (int32_t*)take(TK * 4);
  S.xs = (uint16_t*)take(TK * H * 2);
  S.hh = (uint16_t*)take(TK * I * 2);
  S.hh_lo = (uint16_t*)take(TK * I * 2);
  S.y = (float*)take(TK * H * 4);
  S.groups = (int4*)take((E + TK / 256 + 2) * 16);
  S.ctl = (int32_t*)take(16 * 4);
  return S;
}

// position of column k (0..7) of an 8-column block in P8 order (0 4 1 5 2 6 3 7)
__device__ __forceinline__ int p8pos(int k) { return k < 4 ? 2 * k : 2 * (k - 4) + 1; }

__device__ __forceinline__ float warp_sum_c(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// x (or RMSNorm(h) * gamma rounded to fp16) -> xp in P8 order; one warp per token
__global__ void k_chunk_prologue(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps,
                                 int T, int H, uint16_t* __restrict__ xp) {
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (t >= T) return;
  const uint16_t* xr = x + (size_t)t * H;
  float rn = 1.f;
  if (gamma) {
    float ss = 0.f;
    for (int i = lane; i < H; i += 32) {
      const float v = __half2float(__ushort_as_half(xr[i]));
      ss += v * v;
    }
    ss = warp_sum_c(ss);
    rn = 1.0f / sqrtf(ss / (float)H + eps);
  }
  for (int blk = lane; blk < H / 8; blk += 32) {
    uint16_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = blk * 8 + k;
      uint16_t v = xr[c];
      if (gamma)
        v = __half_as_ushort(__float2half_rn(__half2float(__ushort_as_half(v)) * rn *
                                             __half2float(__ushort_as_half(gamma[c]))));
      o[p8pos(k)] = v;
    }
    uint4 pk;
    pk.x = o[0] | ((uint32_t)o[1] << 16);
    pk.y = o[2] | ((uint32_t)o[3] << 16);
    pk.z = o[4] | ((uint32_t)o[5] << 16);
    pk.w = o[6] | ((uint32_t)o[7] << 16);
    *reinterpret_cast<uint4*>(xp + (size_t)t * H + blk * 8) = pk;
  }
}

// softmax over the E expert logits -> the k largest (lower index on ties) -> renormalise; sigmoid of logit E.
// One warp per token; ids ascending. Also marks the token in its experts' masks.
__global__ void k_chunk_route(const float* __restrict__ logits, int E, int K, int T, int32_t* __restrict__ ids,
                              float* __restrict__ w, float* __restrict__ sg, uint32_t* __restrict__ masks, int TW,
                              int32_t* rec_ids, float* rec_w, float* rec_sg) {
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* lg = logits + (size_t)t * (E + 1);
  constexpr int MAXEPL = 16;
  const int epl = (E + 31) / 32;
  float v[MAXEPL];
#pragma unroll
  for (int i = 0; i < MAXEPL; ++i) {
    const int e = lane * epl + i;
    v[i] = (i < epl && e < E) ? lg[e] : -INFINITY;
  }
  int sel_idx = -1;
  float sel_val = 0.f;
  for (int j = 0; j < K; ++j) {
    float best = -INFINITY;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < MAXEPL; ++i)
      if (v[i] > best) { best = v[i]; bi = i; }
    int be = best == -INFINITY ? 0x7FFFFFFF : lane * epl + bi;
    float m = best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
      if (om > m || (om == m && oe < be)) { m = om; be = oe; }
    }
    if (be == lane * epl + bi && best == m) {
#pragma unroll
      for (int i = 0; i < MAXEPL; ++i)
        if (i == bi) v[i] = -INFINITY;
    }
    if (lane == j) { sel_idx = be; sel_val = m; }
  }
  const float mx = __shfl_sync(0xFFFFFFFFu, sel_val, 0);
  const float ex = lane < K ? __expf(sel_val - mx) : 0.f;
  const float z = warp_sum_c(ex);
  int rank = 0;
  for (int i = 0; i < K; ++i) rank += (__shfl_sync(0xFFFFFFFFu, sel_idx, i) < sel_idx) ? 1 : 0;
  if (lane < K) {
    const float wv = __fdividef(ex, z);
    ids[(size_t)t * K + rank] = sel_idx;
    w[(size_t)t * K + rank] = wv;
    if (rec_ids) { rec_ids[(size_t)t * K + rank] = sel_idx; rec_w[(size_t)t * K + rank] = wv; }
    atomicOr(&masks[(size_t)sel_idx * TW + (t >> 5)], 1u << (t & 31));
  }
  if (lane == 0) {
    const float g = __frcp_rn(1.0f + __expf(-lg[E]));
    sg[t] = g;
    if (rec_sg) rec_sg[t] = g;
  }
}

// One CTA: per-expert token counts from the masks, exclusive scan, the sorted row of every (token, slot), the
// token of every sorted row, and the list of 256-row tile groups (expert, first row, rows); job counters reset.
__global__ void k_chunk_bucket(const uint32_t* __restrict__ masks, int E, int TW, int T, int K,
                               const int32_t* __restrict__ ids, int32_t* __restrict__ slot_of,
                               int32_t* __restrict__ tok_of, int4* __restrict__ groups, int32_t* __restrict__ ctl) {
  __shared__ int cnt[512], off[512], ngrp[512], goff[512];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int q = 0; q < TW; ++q) c += __popc(masks[(size_t)e * TW + q]);
    cnt[e] = c;
    ngrp[e] = (c + 255) / 256;
  }
  __syncthreads();
  if (tid == 0) {
    int o = 0, go = 0;
    for (int e = 0; e < E; ++e) { off[e] = o; o += cnt[e]; goff[e] = go; go += ngrp[e]; }
    ctl[0] = go;                     // number of tile groups
    for (int k = 1; k < 8; ++k) ctl[k] = 0;   // job counters of the GEMM launches
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x)
    for (int g = 0; g < ngrp[e]; ++g)
      groups[goff[e] + g] = make_int4(e, off[e] + g * 256, min(256, cnt[e] - g * 256), 0);
  for (int p = tid; p < T * K; p += blockDim.x) {
    const int t = p / K, e = ids[p];
    int rank = 0;
    const uint32_t* m = masks + (size_t)e * TW;
    for (int q = 0; q < (t >> 5); ++q) rank += __popc(m[q]);
    rank += __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
    const int row = off[e] + rank;
    slot_of[p] = row;
    tok_of[row] = t;
  }
}

// xs[row] = xp[tok_of[row]] (fp16 rows of H); one warp per row
__global__ void k_chunk_gather(const uint16_t* __restrict__ xp, const int32_t* __restrict__ tok_of, int rows, int H,
                               uint16_t* __restrict__ xs) {
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(xp + (size_t)tok_of[r] * H);
  uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)r * H);
  for (int i = lane; i < H / 8; i += 32) dst[i] = src[i];
}

// out[t][r] = sum_j w[t][j] * y[slot(t, j)][r] + sg[t] * ys[t][r] (+ h[t][r]), rounded to fp16 once
__global__ void k_chunk_combine(const float* __restrict__ y, const float* __restrict__ ys,
                                const int32_t* __restrict__ slot_of, const float* __restrict__ w,
                                const float* __restrict__ sg, const uint16_t* __restrict__ resid, int T, int H,
                                int K, uint16_t* __restrict__ out) {
  const size_t n = (size_t)T * H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H), r = (int)(i % H);
    float acc = 0.f;
    for (int j = 0; j < K; ++j) acc += w[(size_t)t * K + j] * y[(size_t)slot_of[(size_t)t * K + j] * H + r];
    acc += sg[t] * ys[i];
    if (resid) acc += __half2float(__ushort_as_half(resid[i]));
    out[i] = __half_as_ushort(__float2half_rn(acc));
  }
}

// ------------------------------------------------------------------------------------------ grouped GEMM
enum : int { GK_ROUTER = 0, GK_SHGU = 1, GK_SHDN = 2, GK_EXGU = 3, GK_EXDN = 4 };

struct GemmArgs {
  GemmLayout G;
  ChunkScratch S;
  int T;
  int phase;            // 1: router + shared gate/up, 2: expert gate/up + shared down, 3: expert down
  uint32_t* status;
  uint64_t timeout_ns;
};

struct Job {
  int kind, m, row0, cnt;   // row0 / cnt: first activation row and rows of this N tile
  const uint8_t* a;         // codes of row 128*m of the matrix
  const uint32_t* sb;       // (s, b) pairs, group-major, already offset by 128*m
  int sb_rows;              // rows of the matrix (stride of the group-major pairs)
  int rowbytes, int8, ktiles;
  const uint16_t* act;      // activations [rows][64*ktiles] fp16 P8
  const uint16_t* act_lo;   // low halves of split activations (down projections: h), else null
  int e;                    // expert (routed kinds)
};

constexpr int GT = 128;                      // threads per GEMM CTA
constexpr int G_A16 = 0;                     // 2 x 16 KB
constexpr int G_ALO = 32768;                 // 2 x 16 KB: low halves of split router weights
constexpr int G_B = 65536;                   // 3 x 32 KB
constexpr int G_CODES = 65536 + 3 * 32768;   // 3 x 8 KB
constexpr int G_SB = G_CODES + 3 * 8192;     // 3 x 512 B
constexpr int G_BAR = G_SB + 3 * 512;        // 3 mbarriers, tmem slot, job slot
constexpr int G_SMEM = G_BAR + 128 + 1024;   // + alignment slack

__device__ bool decode_job(const GemmArgs& g, int j, Job& jb) {
  const GemmLayout& G = g.G;
  const int NT = (g.T + 255) / 256;
  jb.e = 0;
  jb.act_lo = nullptr;
  if (g.phase == 1) {
    const int MTr = G.Mr / 128, MTs = 2 * G.Is / 128;
    if (j < MTr * NT) {
      jb.kind = GK_ROUTER; jb.m = j % MTr; const int nt = j / MTr;
      jb.row0 = nt * 256; jb.cnt = min(256, g.T - jb.row0);
      jb.a = G.gr + (size_t)jb.m * 128 * G.H; jb.sb = G.grs + jb.m * 128; jb.sb_rows = G.Mr;
      jb.rowbytes = G.H; jb.int8 = 1; jb.ktiles = G.H / 64; jb.act = g.S.xp;
      return true;
    }
    j -= MTr * NT;
    if (j < MTs * NT) {
      jb.kind = GK_SHGU; jb.m = j % MTs; const int nt = j / MTs;
      jb.row0 = nt * 256; jb.cnt = min(256, g.T - jb.row0);
      jb.a = G.gsgu + (size_t)jb.m * 128 * G.H; jb.sb = G.gsgus + jb.m * 128; jb.sb_rows = 2 * G.Is;
      jb.rowbytes = G.H; jb.int8 = 1; jb.ktiles = G.H / 64; jb.act = g.S.xp;
      return true;
    }
    return false;
  }
  const int ngroups = g.S.ctl[0];
  if (g.phase == 2) {
    const int MTg = 2 * G.I / 128, MTd = G.H / 128;
    if (j < ngroups * MTg) {
      const int4 gr = g.S.groups[j / MTg];
      jb.kind = GK_EXGU; jb.m = j % MTg; jb.e = gr.x; jb.row0 = gr.y; jb.cnt = gr.z;
      jb.a = G.gegu + gr.x * G.gegu_expert + (size_t)jb.m * 128 * (G.H / 2);
      jb.sb = G.gegus + gr.x * G.gegus_expert + jb.m * 128; jb.sb_rows = 2 * G.I;
      jb.rowbytes = G.H / 2; jb.int8 = 0; jb.ktiles = G.H / 64; jb.act = g.S.xs;
      return true;
    }
    j -= ngroups * MTg;
    // down projections take N tiles of at most 128 tokens: the low halves of h share the B stage
    const int NT128 = (g.T + 127) / 128;
    if (j < MTd * NT128) {
      jb.kind = GK_SHDN; jb.m = j % MTd; const int nt = j / MTd;
      jb.row0 = nt * 128; jb.cnt = min(128, g.T - jb.row0);
      jb.a = G.gsdn + (size_t)jb.m * 128 * G.Is; jb.sb = G.gsdns + jb.m * 128; jb.sb_rows = G.H;
      jb.rowbytes = G.Is; jb.int8 = 1; jb.ktiles = G.Is / 64; jb.act = g.S.hs; jb.act_lo = g.S.hs_lo;
      return true;
    }
    return false;
  }
  const int MTd = G.H / 128;
  // each group of up to 256 rows in two halves of up to 128; both halves of a weight tile are consecutive jobs
  if (j < ngroups * MTd * 2) {
    const int4 gr = g.S.groups[j / (2 * MTd)];
    const int half = j & 1;
    jb.kind = GK_EXDN; jb.m = (j % (2 * MTd)) >> 1; jb.e = gr.x;
    jb.row0 = gr.y + 128 * half; jb.cnt = max(0, min(128, gr.z - 128 * half));
    jb.a = G.gedn + gr.x * G.gedn_expert + (size_t)jb.m * 128 * (G.I / 2);
    jb.sb = G.gedns + gr.x * G.gedns_expert + jb.m * 128; jb.sb_rows = G.H;
    jb.rowbytes = G.I / 2; jb.int8 = 0; jb.ktiles = G.I / 64; jb.act = g.S.hh; jb.act_lo = g.S.hh_lo;
    return true;
  }
  return false;
}

// asynchronous loads of K-tile kt of a job into stage st: 128 rows of codes, their (s, b) pairs, N activation
// rows (zero rows beyond cnt) in the swizzled layout
__device__ __forceinline__ void load_ktile(uint8_t* smem, const Job& jb, int kt, int st, int N) {
  const int tid = threadIdx.x;
  uint8_t* codes = smem + G_CODES + st * 8192;
  const int cb = jb.int8 ? 64 : 32;   // code bytes per row per K-tile
  for (int q = tid; q < 128 * cb / 16; q += GT) {
    const int row = q / (cb / 16), part = q % (cb / 16);
    cp_async16(codes + row * cb + part * 16, jb.a + (size_t)row * jb.rowbytes + (size_t)kt * cb + part * 16, 16);
  }
  if (tid < 32)
    cp_async16(smem + G_SB + st * 512 + tid * 16, jb.sb + (size_t)kt * jb.sb_rows + tid * 4, 16);
  uint8_t* B = smem + G_B + st * 32768;
  const int kdim = jb.ktiles * 64;
  for (int q = tid; q < N * 8; q += GT) {
    const int n = q >> 3, c = q & 7;
    const bool valid = n < jb.cnt;
    const uint16_t* src = jb.act + (size_t)(jb.row0 + (valid ? n : 0)) * kdim + kt * 64 + c * 8;
    cp_async16(B + sw128_off(n, c), src, valid ? 16 : 0);
    if (jb.act_lo) cp_async16(B + 16384 + sw128_off(n, c), src - jb.act + jb.act_lo, valid ? 16 : 0);
  }
}

// K-tile codes of stage st -> split fp16 weights in the A buffers ab (thread = row). With w = s*q + b formed in
// fp32 (s*q is exact, one rounding for the sum): hi = RN_fp16(w), lo = RN_fp16(4096 (w - hi)); w - hi is exact
// in fp32, and the scaled low half stays clear of fp16 subnormals. hi x + lo x / 4096 carries w to ~2^-22.
template <bool INT8>
__device__ __forceinline__ void dequant_ktile(uint8_t* smem, int st, int ab) {
  const int r = threadIdx.x;
  const uint8_t* codes = smem + G_CODES + st * 8192;
  const uint32_t sbw = *reinterpret_cast<const uint32_t*>(smem + G_SB + st * 512 + r * 4);
  const uint32_t s2 = (sbw & 0xFFFFu) * 0x10001u;   // (s, s)
  const float bf = __half2float(__ushort_as_half((unsigned short)(sbw >> 16)));
  const __half2 k1024 = __float2half2_rn(1024.0f), k16 = __float2half2_rn(0.0625f), k64 = __float2half2_rn(-64.0f);
  const uint32_t neg1 = 0xBC00BC00u;                // (-1, -1)
  const float2 k4096 = make_float2(4096.0f, 4096.0f);
  uint8_t* A = smem + G_A16 + ab * 16384;
  uint8_t* Alo = smem + G_ALO + ab * 16384;
#pragma unroll 4
  for (int c = 0; c < 8; ++c) {
    uint32_t v[4];
    if (INT8) {
      const uint2 w = *reinterpret_cast<const uint2*>(codes + r * 64 + c * 8);
      int8_block_pairs(w.x, w.y, v);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + r * 32 + c * 4);
      int4_word_pairs(w, v);
    }
    uint32_t oh[4], ol[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = *reinterpret_cast<const __half2*>(&v[k]);
      // exact codes: 1024 + q -> q; 1024 + 16 q (odd int4 pairs) -> q
      const __half2 q = (!INT8 && (k & 1)) ? __hfma2(h, k16, k64) : __hsub2(h, k1024);
      const uint32_t qu = *reinterpret_cast<const uint32_t*>(&q);
      const float p0 = fmix_lo(s2, qu, bf), p1 = fmix_hi(s2, qu, bf);
      const __half2 hi = __floats2half2_rn(p0, p1);
      const uint32_t hu = *reinterpret_cast<const uint32_t*>(&hi);
      const float2 d = __fmul2_rn(make_float2(fmix_lo(hu, neg1, p0), fmix_hi(hu, neg1, p1)), k4096);
      const __half2 lo = __floats2half2_rn(d.x, d.y);
      oh[k] = hu;
      ol[k] = *reinterpret_cast<const uint32_t*>(&lo);
    }
    *reinterpret_cast<uint4*>(A + sw128_off(r, c)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    *reinterpret_cast<uint4*>(Alo + sw128_off(r, c)) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
  }
}

// 16 accumulator columns of this warp's rows: hi sum + low sum / 4096
__device__ __forceinline__ void tmem_ld_split(uint32_t taddr, float (&v)[16]) {
  float l[16];
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + 256, l);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = fmaf(l[i], 1.0f / 4096.0f, v[i]);
}

__device__ __forceinline__ float silu_c(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__global__ void __launch_bounds__(GT, 1) k_chunk_gemm(GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + G_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + G_BAR + 32);
  int* jslot = reinterpret_cast<int*>(smem + G_BAR + 48);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G_BAR + 64);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GemmLayout& G = g.G;
  const int njobs_max = 1 << 30;

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&mbar[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // columns [0, 256): sum of hi products; [256, 512): sum of products with a low half (scaled by 4096)
  if (warp == 0) { tmem_alloc(tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  uint32_t gk = 0;   // K-tiles this CTA has issued MMAs for (selects stage and mbarrier phase)
  // wait for the MMAs of global K-tile index k to complete
  auto wait_mma = [&](uint32_t k) {
    if (!mbar_wait(&mbar[k % 3], (k / 3) & 1u, g.timeout_ns)) {
      atomicOr(g.status, 256u);
      *abort_flag = 1;
    }
  };

  for (int it = 0; it < njobs_max; ++it) {
    if (tid == 0) *jslot = atomicAdd(&g.S.ctl[g.phase], 1);
    __syncthreads();
    const int j = *jslot;
    Job jb;
    if (*abort_flag || !decode_job(g, j, jb)) break;
    if (jb.cnt <= 0) {   // empty half of a down-projection group
      __syncthreads();
      continue;
    }
    const int N = (jb.cnt + 15) & ~15;
    const int KT = jb.ktiles;
    const uint32_t base = gk;   // global index of this job's first K-tile
    // stages of K-tiles base and base+1 were last read by MMAs base-3 and base-2: wait for them
    if (base >= 3) wait_mma(base - 3);
    load_ktile(smem, jb, 0, base % 3, N);
    cp_async_commit();
    if (KT > 1) {
      if (base + 1 >= 3) wait_mma(base - 2);
      load_ktile(smem, jb, 1, (base + 1) % 3, N);
    }
    cp_async_commit();
    for (int kt = 0; kt < KT; ++kt) {
      const uint32_t k = base + kt;
      cp_async_wait<1>();
      __syncthreads();
      if (k >= 2) wait_mma(k - 2);   // A buffer k&1 was read by MMA k-2
      if (jb.int8) dequant_ktile<true>(smem, k % 3, k & 1);
      else dequant_ktile<false>(smem, k % 3, k & 1);
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0 && !*abort_flag) {
        tc_fence_after();
        const uint32_t idesc = umma_idesc_f16(128, N);
        const uint32_t a0 = smem_u32(smem + G_A16 + (k & 1) * 16384), b0 = smem_u32(smem + G_B + (k % 3) * 32768);
        const uint32_t l0 = smem_u32(smem + G_ALO + (k & 1) * 16384);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t acc = (kt > 0 || ks > 0) ? 1u : 0u;
          umma_f16(tmem, umma_desc_sw128(a0 + 32 * ks), umma_desc_sw128(b0 + 32 * ks), idesc, acc);
          umma_f16(tmem + 256, umma_desc_sw128(l0 + 32 * ks), umma_desc_sw128(b0 + 32 * ks), idesc, acc);
          if (jb.act_lo)
            umma_f16(tmem + 256, umma_desc_sw128(a0 + 32 * ks), umma_desc_sw128(b0 + 16384 + 32 * ks), idesc, 1u);
        }
        umma_commit(&mbar[k % 3]);
      }
      if (kt + 2 < KT) {
        if (k + 2 >= 3) wait_mma(k - 1);   // stage (k+2)%3 was read by MMA k-1
        load_ktile(smem, jb, kt + 2, (k + 2) % 3, N);
      }
      cp_async_commit();
    }
    gk = base + KT;
    wait_mma(gk - 1);
    tc_fence_after();
    if (*abort_flag) break;
    // ---- epilogue: thread = accumulator row (TMEM lane), columns = the tile's tokens
    const int r = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const bool swiglu = jb.kind == GK_SHGU || jb.kind == GK_EXGU;
    float* xch = reinterpret_cast<float*>(smem + G_B);   // up rows for SwiGLU: [64][N + 1]
    if (swiglu && warp >= 2) {
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld_split(trow + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) xch[(r - 64) * (N + 1) + c0 + i] = v[i];
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!swiglu || warp < 2) {
      for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld_split(trow + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          if (n >= jb.cnt) continue;
          const size_t row = (size_t)(jb.row0 + n);
          if (jb.kind == GK_ROUTER) {
            const int er = jb.m * 128 + r;
            if (er <= G.E) g.S.logits[row * (G.E + 1) + er] = v[i];
          } else if (jb.kind == GK_SHDN) {
            g.S.ys[row * G.H + jb.m * 128 + r] = v[i];
          } else if (jb.kind == GK_EXDN) {
            g.S.y[row * G.H + jb.m * 128 + r] = v[i];
          } else {
            const float h = silu_c(v[i]) * xch[r * (N + 1) + n];
            const int u = jb.m * 64 + r;
            const int pos = (u & ~7) + ((u & 7) < 4 ? 2 * (u & 7) : 2 * ((u & 7) - 4) + 1);
            const __half hh = __float2half_rn(h);
            const uint16_t hv = __half_as_ushort(hh);
            const uint16_t lv = __half_as_ushort(__float2half_rn((h - __half2float(hh)) * 4096.0f));
            if (jb.kind == GK_SHGU) {
              g.S.hs[row * G.Is + pos] = hv;
              g.S.hs_lo[row * G.Is + pos] = lv;
            } else {
              g.S.hh[row * G.I + pos] = hv;
              g.S.hh_lo[row * G.I + pos] = lv;
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t chunk_forward(const MoeLayout& L, const GemmLayout& G, const ChunkScratch& S, int num_sms,
                          const uint16_t* x, uint16_t* out, int T, const uint16_t* gamma, float eps,
                          int32_t* rec_ids, float* rec_w, float* rec_sg, uint32_t* status, uint64_t timeout_ns,
                          cudaStream_t st, int* launches) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_chunk_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int E = L.E, K = L.K, H = L.H, TW = (T + 31) / 32;
  int n = 0;
  cudaError_t e = cudaMemsetAsync(S.ctl, 0, 16 * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(S.masks, 0, (size_t)E * TW * 4, st);
  if (e != cudaSuccess) return e;
  k_chunk_prologue<<<(T + 7) / 8, 256, 0, st>>>(x, gamma, eps, T, H, S.xp);
  ++n;
  GemmArgs ga{G, S, T, 1, status, timeout_ns};
  const int NT = (T + 255) / 256;
  const int jobs1 = (G.Mr / 128 + 2 * G.Is / 128) * NT;
  k_chunk_gemm<<<jobs1 < num_sms ? jobs1 : num_sms, GT, G_SMEM, st>>>(ga);
  ++n;
  k_chunk_route<<<(T + 7) / 8, 256, 0, st>>>(S.logits, E, K, T, S.ids, S.w, S.sg, S.masks, TW, rec_ids, rec_w,
                                              rec_sg);
  ++n;
  k_chunk_bucket<<<1, 512, 0, st>>>(S.masks, E, TW, T, K, S.ids, S.slot_of, S.tok_of, S.groups, S.ctl);
  ++n;
  k_chunk_gather<<<(T * K + 7) / 8, 256, 0, st>>>(S.xp, S.tok_of, T * K, H, S.xs);
  ++n;
  ga.phase = 2;
  k_chunk_gemm<<<num_sms, GT, G_SMEM, st>>>(ga);
  ++n;
  ga.phase = 3;
  k_chunk_gemm<<<num_sms, GT, G_SMEM, st>>>(ga);
  ++n;
  const size_t tot = (size_t)T * H;
  const int cg = (int)((tot + 255) / 256 < 65536 ? (tot + 255) / 256 : 65536);
  k_chunk_combine<<<cg, 256, 0, st>>>(S.y, S.ys, S.slot_of, S.w, S.sg, gamma ? x : nullptr, T, H, K, out);
  ++n;
  if (launches) *launches = n;
  return cudaGetLastError();
}

}  // namespace moe
