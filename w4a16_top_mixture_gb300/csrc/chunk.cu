// Prompt-chunk path of the W4A16 routed-MoE block (T > 16): weight repack into the tiled GEMM layout, routing /
// bucketing / gather kernels, the final combine and the launch sequence. The GEMM kernel is in chunk_gemm.cu.
// See chunk.cuh for the layouts.
#include <cuda_fp16.h>
#include <stdint.h>
#include <utility>

#include "chunk.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {

static size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

// Every kernel of the chunk path is launched programmatic-dependent: its CTAs may become resident while the
// previous kernel on the stream still runs (once every CTA of that one has run launch_dependents or exited), and
// each kernel runs griddepcontrol.wait before it reads anything an earlier kernel writes, or writes anything an
// earlier kernel reads. Only launch latency and set-up overlap; no data is read early. Data an earlier kernel
// wrote is read through L2 (ld.global.cg): while launches overlap, nothing is taken to keep a line of it that an
// earlier launch left in this SM's L1 from being stale.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*k)(KArgs...), int grid, int block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

size_t gemm_store_bytes(const MoeLayout& L) {
  const size_t H = L.H, E = L.E, I = L.I, Is = L.Is, Mr = ((L.E + 1 + 127) / 128) * 128;
  size_t b = 0;
  b += al256((Mr / 128) * (H / 64) * GEMM_BLK8);            // router
  b += al256((2 * Is / 128) * (H / 64) * GEMM_BLK8);        // shared gate/up
  b += al256((H / 128) * (Is / 64) * GEMM_BLK8);            // shared down
  b += al256(E * (2 * I / 128) * (H / 64) * GEMM_BLK4);     // expert gate/up
  b += al256(E * (H / 128) * (I / 64) * GEMM_BLK4);         // expert down
  return b;
}

GemmLayout gemm_layout_carve(const MoeLayout& L, uint8_t* base) {
  GemmLayout G;
  G.H = L.H; G.E = L.E; G.K = L.K; G.I = L.I; G.Is = L.Is;
  G.Mr = ((L.E + 1 + 127) / 128) * 128;
  const size_t H = L.H, E = L.E, I = L.I, Is = L.Is, Mr = G.Mr;
  uint8_t* p = base;
  auto take = [&](size_t n) { uint8_t* r = p; p += al256(n); return r; };
  G.gr = take((Mr / 128) * (H / 64) * GEMM_BLK8);
  G.gsgu = take((2 * Is / 128) * (H / 64) * GEMM_BLK8);
  G.gsdn = take((H / 128) * (Is / 64) * GEMM_BLK8);
  G.gegu_expert = (2 * I / 128) * (H / 64) * GEMM_BLK4;
  G.gedn_expert = (H / 128) * (I / 64) * GEMM_BLK4;
  G.gegu = take(E * G.gegu_expert);
  G.gedn = take(E * G.gedn_expert);
  return G;
}

// One thread per (batch, row, K-tile): copies the row's 64 codes of that tile (32 or 64 bytes) and its (s, b)
// pair into the tile block. rowmode 0 keeps the row index; 1 / 2 place row r of a gate / up matrix into band
// r/64 at position (0 | 64) + r%64. int8 rows get the P8 byte order inside each 8-byte block. The GEMM forms
// s * q in fp16 (as an exact pair of halves), so a scale that is not finite, or whose product with the largest
// code reaches fp16's largest finite value, sets *range_bad.
__global__ void k_gemm_tiles(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                             const uint16_t* __restrict__ b, int nbatch, int nrows, int cols, int int8,
                             size_t src_q_batch, size_t src_sb_batch, uint8_t* __restrict__ dst,
                             size_t dst_batch, int rowmode, uint32_t* __restrict__ range_bad) {
  const int KT = cols / 64, cb = int8 ? 64 : 32, blk = int8 ? GEMM_BLK8 : GEMM_BLK4;
  const int rowbytes = int8 ? cols : cols / 2;
  const size_t n = (size_t)nbatch * nrows * KT;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int kt = (int)(i % KT);
    const size_t t = i / KT;
    const int r = (int)(t % nrows);
    const int bt = (int)(t / nrows);
    const int dr = rowmode == 0 ? r : (r / 64) * 128 + (rowmode == 2 ? 64 : 0) + r % 64;
    const int mt = dr / 128, rr = dr % 128;
    uint8_t* tile = dst + bt * dst_batch + ((size_t)mt * KT + kt) * blk;
    const uint8_t* src = q + bt * src_q_batch + (size_t)r * rowbytes + (size_t)kt * cb;
    uint8_t* dc = tile + (size_t)rr * cb;
    if (int8) {
      const int pos[8] = {0, 1, 4, 5, 2, 3, 6, 7};   // destination byte j holds column pos[j]
      for (int b8 = 0; b8 < 8; ++b8)
#pragma unroll
        for (int j = 0; j < 8; ++j) dc[b8 * 8 + j] = src[b8 * 8 + pos[j]];
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) dc[j] = src[j];
    }
    const size_t si = bt * src_sb_batch + (size_t)r * KT + kt;
    *reinterpret_cast<uint32_t*>(tile + 128 * cb + rr * 4) = (uint32_t)s[si] | ((uint32_t)b[si] << 16);
    const float sv = __half2float(__ushort_as_half(s[si]));
    if (!(fabsf(sv) * (int8 ? 255.0f : 15.0f) < 65504.0f)) atomicOr(range_bad, 1u);
  }
}

static int grid_for_n(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 65535 * 8) g = 65535 * 8;
  return g < 1 ? 1 : (int)g;
}

cudaError_t gemm_repack(const RepackSrc& w, const GemmLayout& G, uint32_t* range_bad, cudaStream_t st) {
  const int H = G.H, E = G.E, I = G.I, Is = G.Is;
  // the router's padding rows stay zero: codes 0, s = b = 0
  cudaError_t e = cudaMemsetAsync(G.gr, 0, (size_t)(G.Mr / 128) * (H / 64) * GEMM_BLK8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(range_bad, 0, 4, st);
  if (e != cudaSuccess) return e;
  auto tiles = [&](const uint8_t* q, const uint16_t* s, const uint16_t* b, int nbatch, int nrows, int cols,
                   int int8, size_t sqb, size_t ssb, uint8_t* dst, size_t db, int rowmode) {
    const size_t n = (size_t)nbatch * nrows * (cols / 64);
    k_gemm_tiles<<<grid_for_n(n), 256, 0, st>>>(q, s, b, nbatch, nrows, cols, int8, sqb, ssb, dst, db, rowmode,
                                                 range_bad);
  };
  tiles(w.router_q, w.router_s, w.router_b, 1, E + 1, H, 1, 0, 0, G.gr, 0, 0);
  tiles(w.sh_gate_q, w.sh_gate_s, w.sh_gate_b, 1, Is, H, 1, 0, 0, G.gsgu, 0, 1);
  tiles(w.sh_up_q, w.sh_up_s, w.sh_up_b, 1, Is, H, 1, 0, 0, G.gsgu, 0, 2);
  tiles(w.sh_down_q, w.sh_down_s, w.sh_down_b, 1, H, Is, 1, 0, 0, G.gsdn, 0, 0);
  tiles(w.exp_gate_q, w.exp_gate_s, w.exp_gate_b, E, I, H, 0, (size_t)I * (H / 2), (size_t)I * (H / 64), G.gegu,
        G.gegu_expert, 1);
  tiles(w.exp_up_q, w.exp_up_s, w.exp_up_b, E, I, H, 0, (size_t)I * (H / 2), (size_t)I * (H / 64), G.gegu,
        G.gegu_expert, 2);
  tiles(w.exp_down_q, w.exp_down_s, w.exp_down_b, E, H, I, 0, (size_t)H * (I / 2), (size_t)H * (I / 64), G.gedn,
        G.gedn_expert, 0);
  return cudaGetLastError();
}

size_t chunk_scratch_bytes(const MoeLayout& L, int Tm) {
  const size_t H = L.H, E = L.E, K = L.K, I = L.I, Is = L.Is, T = Tm, TK = (size_t)Tm * L.K;
  const size_t TW = (T + 31) / 32;
  size_t b = 0;
  b += al256(T * H * 2) + al256(ROUTER_SPLIT * T * logit_stride((int)E) * 4);
  b += al256(T * Is * 2) * 2 + al256(T * H * 4);
  b += al256(T * K * 4) * 2 + al256(T * 4) + al256(E * TW * 4) + al256(T * K * 4) + al256(TK * 4);
  b += al256(TK * H * 2);
  b += al256(TK * I * 2) * 2 + al256(TK * H * 4);
  b += al256((E + TK / CHUNK_NT + 2) * 16) + al256(16 * 4);
  b += al256(T * GSUM_COLS * 2) * 2 + al256(TK * GSUM_COLS * 2) * 2;
  return b;
}

ChunkScratch chunk_scratch_carve(const MoeLayout& L, int Tm, uint8_t* base) {
  const size_t H = L.H, E = L.E, K = L.K, I = L.I, Is = L.Is, T = Tm, TK = (size_t)Tm * L.K;
  const size_t TW = (T + 31) / 32;
  uint8_t* p = base;
  auto take = [&](size_t n) { uint8_t* r = p; p += al256(n); return r; };
  ChunkScratch S;
  S.xp = (uint16_t*)take(T * H * 2);
  S.logits = (float*)take(ROUTER_SPLIT * T * logit_stride((int)E) * 4);
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
  S.groups = (int4*)take((E + TK / CHUNK_NT + 2) * 16);
  S.ctl = (int32_t*)take(16 * 4);
  S.gs_xp = (uint16_t*)take(T * GSUM_COLS * 2);
  S.gs_hs = (uint16_t*)take(T * GSUM_COLS * 2);
  S.gs_xs = (uint16_t*)take(TK * GSUM_COLS * 2);
  S.gs_hh = (uint16_t*)take(TK * GSUM_COLS * 2);
  return S;
}

cudaError_t chunk_make_maps(const MoeLayout& L, const ChunkScratch& S, int Tm, ChunkMaps* out) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fp) return e != cudaSuccess ? e : cudaErrorNotSupported;
    encode = reinterpret_cast<EncodeFn>(fp);
  }
  const int TK = Tm * L.K;
  struct Buf { const uint16_t* p; int rows, cols; };
  const Buf bufs[CM_COUNT] = {{S.xp, Tm, L.H},          {S.xs, TK, L.H},          {S.hs, Tm, L.Is},
                              {S.hs_lo, Tm, L.Is},      {S.hh, TK, L.I},          {S.hh_lo, TK, L.I},
                              {S.gs_xp, Tm, GSUM_COLS}, {S.gs_xs, TK, GSUM_COLS}, {S.gs_hs, Tm, GSUM_COLS},
                              {S.gs_hh, TK, GSUM_COLS}};
  const cuuint32_t boxrows[CM_BOXES] = {16, 32, CHUNK_NT};
  for (int b = 0; b < CM_COUNT; ++b)
    for (int v = 0; v < CM_BOXES; ++v) {
      const cuuint64_t dims[2] = {(cuuint64_t)bufs[b].cols, (cuuint64_t)bufs[b].rows};
      const cuuint64_t strides[1] = {(cuuint64_t)bufs[b].cols * 2};
      const cuuint32_t box[2] = {64, boxrows[v]};
      const cuuint32_t estr[2] = {1, 1};
      const CUresult r = encode(&out->m[b][v], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)bufs[b].p, dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
  return cudaSuccess;
}

// position of column k (0..7) of an 8-column block in P8 order (0 4 1 5 2 6 3 7)
__device__ __forceinline__ int p8pos(int k) { return k < 4 ? 2 * k : 2 * (k - 4) + 1; }

__device__ __forceinline__ float warp_sum_c(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// the group-sum row entries of group g: the fp32 sum as fp16 hi + fp16 remainder
__device__ __forceinline__ void put_gsum(uint16_t* row, int g, float v) {
  const __half hi = __float2half_rn(v);
  const __half lo = __float2half_rn(v - __half2float(hi));
  *reinterpret_cast<uint32_t*>(row + 2 * g) = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
}

// x (or RMSNorm(h) * gamma rounded to fp16) -> xp in P8 order, and the sum of each 64-column group of the
// written values -> the token's group-sum row. PRO_WPT warps per token, each taking every PRO_WPT-th run of 32
// 8-column blocks (one 16-byte load per lane); the eight blocks of a group sit on eight neighbouring lanes. With
// gamma, the token's first warp forms 1 / RMS (the lane-strided sum of squares, then a butterfly) for all four.
constexpr int PRO_WPT = 4;
constexpr int PRO_TPC = 2;   // tokens per CTA (PRO_WPT * PRO_TPC warps)
__global__ void __launch_bounds__(PRO_WPT * PRO_TPC * 32)
k_chunk_prologue(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps, int T, int H,
                 uint16_t* __restrict__ xp, uint16_t* __restrict__ gs_xp, uint32_t* __restrict__ masks,
                 int nmask) {
  __shared__ float rn_s[PRO_TPC];
  pdl_wait();
  pdl_release();
  // the routing's expert masks start empty
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nmask; i += gridDim.x * blockDim.x) masks[i] = 0u;
  const int wt = threadIdx.x >> 5, lane = threadIdx.x & 31, tl = wt / PRO_WPT, part = wt % PRO_WPT;
  const int t = blockIdx.x * PRO_TPC + tl;
  const bool live = t < T;
  const uint16_t* xr = x + (size_t)t * H;
  float rn = 1.f;
  if (gamma) {
    if (live && part == 0) {
      float ss = 0.f;
#pragma unroll 8
      for (int i = lane; i < H; i += 32) {
        const float v = __half2float(__ushort_as_half(__ldcg(xr + i)));
        ss += v * v;
      }
      ss = warp_sum_c(ss);
      if (lane == 0) rn_s[tl] = 1.0f / sqrtf(ss / (float)H + eps);
    }
    __syncthreads();
    rn = rn_s[tl];
  }
  if (!live) return;
  const int nblk = H / 8;
#pragma unroll 2
  for (int base = part * 32; base < nblk; base += 32 * PRO_WPT) {
    const int blk = base + lane;
    const bool on = blk < nblk;   // the same for the eight lanes of a group
    const uint4 raw = on ? __ldcg(reinterpret_cast<const uint4*>(xr + blk * 8)) : make_uint4(0, 0, 0, 0);
    const uint4 graw = (gamma && on) ? *reinterpret_cast<const uint4*>(gamma + blk * 8) : make_uint4(0, 0, 0, 0);
    const uint16_t* h8 = reinterpret_cast<const uint16_t*>(&raw);
    const uint16_t* g8 = reinterpret_cast<const uint16_t*>(&graw);
    uint16_t o[8];
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint16_t v = h8[k];
      if (gamma)
        v = __half_as_ushort(__float2half_rn(__half2float(__ushort_as_half(v)) * rn * __half2float(__ushort_as_half(g8[k]))));
      o[p8pos(k)] = v;
      sum += __half2float(__ushort_as_half(v));
    }
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
    if (on) {
      if ((blk & 7) == 0) put_gsum(gs_xp + (size_t)t * GSUM_COLS, blk >> 3, sum);
      uint4 pk;
      pk.x = o[0] | ((uint32_t)o[1] << 16);
      pk.y = o[2] | ((uint32_t)o[3] << 16);
      pk.z = o[4] | ((uint32_t)o[5] << 16);
      pk.w = o[6] | ((uint32_t)o[7] << 16);
      *reinterpret_cast<uint4*>(xp + (size_t)t * H + blk * 8) = pk;
    }
  }
}

// softmax over the E expert logits -> the k largest (lower index on ties) -> renormalise; sigmoid of logit E.
// One warp per token; ids ascending. Also marks the token in its experts' masks. EPL: logits per lane,
// 32 * EPL >= E. The ids are below E whatever the logits hold (NaN and infinities included), so the masks and
// everything indexed by an id stay in bounds.
template <int EPL>
__global__ void k_chunk_route(const float* __restrict__ logits, int np, int E, int K, int T,
                              int32_t* __restrict__ ids, float* __restrict__ w, float* __restrict__ sg,
                              uint32_t* __restrict__ masks, int TW, int32_t* rec_ids, float* rec_w, float* rec_sg) {
  pdl_wait();
  pdl_release();
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (t >= T) return;
  // the logits: the router GEMM's np partial sums, added in part order. Rows are logit_stride(E) floats, so
  // with E a multiple of 128 each lane's EPL logits are whole float4s (all loads issued before the adds)
  const int LS = logit_stride(E);
  const size_t pstride = (size_t)T * LS;
  const float* lg = logits + (size_t)t * LS;
  uint32_t key[EPL];
  if (EPL % 4 == 0 && E == 32 * EPL) {
    constexpr int Q = EPL / 4 > 0 ? EPL / 4 : 1;
    float4 v[ROUTER_SPLIT][Q];
#pragma unroll
    for (int p = 0; p < ROUTER_SPLIT; ++p)
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (p < np) v[p][q] = __ldcg(reinterpret_cast<const float4*>(lg + p * pstride + lane * EPL) + q);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      float4 a = v[0][q];
#pragma unroll
      for (int p = 1; p < ROUTER_SPLIT; ++p)
        if (p < np) { a.x += v[p][q].x; a.y += v[p][q].y; a.z += v[p][q].z; a.w += v[p][q].w; }
      key[4 * q] = topk_key(a.x);
      key[4 * q + 1] = topk_key(a.y);
      key[4 * q + 2] = topk_key(a.z);
      key[4 * q + 3] = topk_key(a.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      float v = 0.f;
      if (e < E) {
        v = __ldcg(lg + e);
        for (int p = 1; p < np; ++p) v += __ldcg(lg + p * pstride + e);
      }
      key[i] = e < E ? topk_key(v) : 0u;
    }
  }
  int sel_idx;
  uint32_t sel_key;
  warp_topk_keys<EPL>(key, K, sel_idx, sel_key);
  const float sel_val = topk_logit(sel_key);
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
    float gl = __ldcg(lg + E);
    for (int p = 1; p < np; ++p) gl += __ldcg(lg + p * pstride + E);
    const float g = __frcp_rn(1.0f + __expf(-gl));
    sg[t] = g;
    if (rec_sg) rec_sg[t] = g;
  }
}

// One CTA per expert e (BUCKET_THREADS threads). Every CTA counts the tokens of every expert from the masks
// (thread = expert) and reduces: its expert's first sorted row (the tokens of the experts before it), its first
// row tile, and, in CTA 0, the launch's row-tile count (ctl[0]) and widest tile (ctl[1]). The CTA then writes its
// expert's row tiles (expert, first row, rows <= CHUNK_NT), and for each of its tokens, in token order, the token
// of the sorted row (tok_of) and the sorted row of the (token, slot) pair (slot_of). Tokens of an expert keep
// their order; the result is the same whatever the grid.
constexpr int BUCKET_THREADS = 256;
__global__ void __launch_bounds__(BUCKET_THREADS, 1) k_chunk_bucket(const uint32_t* __restrict__ masks, int E, int TW,
                                                                 int T, int K, const int32_t* __restrict__ ids,
                                                                 int32_t* __restrict__ slot_of,
                                                                 int32_t* __restrict__ tok_of,
                                                                 int4* __restrict__ groups,
                                                                 int32_t* __restrict__ ctl) {
  __shared__ int red[4][BUCKET_THREADS / 32];
  __shared__ int wpre[BUCKET_THREADS / 32];
  pdl_wait();
  pdl_release();
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = BUCKET_THREADS / 32;
  // every expert's count: the experts before e (rows and tiles), the totals
  int before = 0, gbefore = 0, gtot = 0, wide = 0;
  for (int x = tid; x < E; x += BUCKET_THREADS) {
    const uint32_t* m = masks + (size_t)x * TW;
    int c = 0;
#pragma unroll 8
    for (int q = 0; q < TW; ++q) c += __popc(__ldcg(m + q));
    const int ng = (c + CHUNK_NT - 1) / CHUNK_NT;
    if (x < e) { before += c; gbefore += ng; }
    gtot += ng;
    wide = max(wide, min(c, CHUNK_NT));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xFFFFFFFFu, before, o);
    gbefore += __shfl_xor_sync(0xFFFFFFFFu, gbefore, o);
    gtot += __shfl_xor_sync(0xFFFFFFFFu, gtot, o);
    wide = max(wide, __shfl_xor_sync(0xFFFFFFFFu, wide, o));
  }
  if (lane == 0) { red[0][warp] = before; red[1][warp] = gbefore; red[2][warp] = gtot; red[3][warp] = wide; }
  __syncthreads();
  int off = 0, goff = 0;
  {
    int gt = 0, wd = 0;
    for (int w = 0; w < NW; ++w) { off += red[0][w]; goff += red[1][w]; gt += red[2][w]; wd = max(wd, red[3][w]); }
    if (e == 0 && tid == 0) { ctl[0] = gt; ctl[1] = wd; }
  }
  // this expert's tokens: words of its mask in passes of BUCKET_THREADS / 4 words, four threads a word (8 bits
  // each); a block-wide scan of the words' counts gives each token's rank
  const uint32_t* m = masks + (size_t)e * TW;
  int carry = 0;   // tokens of the expert in earlier passes
  for (int w0 = 0; w0 < TW; w0 += BUCKET_THREADS / 4) {
    const int q = w0 + (tid >> 2), sub = tid & 3;
    const uint32_t word = q < TW ? __ldcg(m + q) : 0u;
    const uint32_t bits = (word >> (8 * sub)) & 0xFFu;
    // inclusive scan of the per-thread counts over the block (thread order = token order)
    int v = __popc(bits), incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) wpre[warp] = incl;
    __syncthreads();
    int wbase = 0, ptot = 0;
    for (int w = 0; w < NW; ++w) { wbase += w < warp ? wpre[w] : 0; ptot += wpre[w]; }
    int rank = carry + wbase + incl - v;
    for (uint32_t r = bits; r != 0u; r &= r - 1u) {
      const int t = 32 * q + 8 * sub + (__ffs(r) - 1);
      const int row = off + rank++;
      tok_of[row] = t;
      for (int j = 0; j < K; ++j)
        if (__ldcg(ids + (size_t)t * K + j) == e) slot_of[(size_t)t * K + j] = row;
    }
    carry += ptot;
    __syncthreads();   // wpre is rewritten by the next pass
  }
  // the expert's row tiles
  for (int g = tid; g * CHUNK_NT < carry; g += BUCKET_THREADS)
    groups[goff + g] = make_int4(e, off + g * CHUNK_NT, min(CHUNK_NT, carry - g * CHUNK_NT), 0);
}

// xs[row] = xp[tok_of[row]] (fp16 rows of H) and its group sums; one warp per row
__global__ void k_chunk_gather(const uint16_t* __restrict__ xp, const uint16_t* __restrict__ gs_xp,
                               const int32_t* __restrict__ tok_of, int rows, int H, uint16_t* __restrict__ xs,
                               uint16_t* __restrict__ gs_xs) {
  pdl_wait();
  pdl_release();
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int t = __ldcg(tok_of + r);
  const uint4* src = reinterpret_cast<const uint4*>(xp + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)r * H);
  // eight 16-byte loads a lane in flight before the stores
  for (int b0 = 0; b0 < H / 8; b0 += 256) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = b0 + k * 32 + lane;
      v[k] = i < H / 8 ? __ldcg(src + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = b0 + k * 32 + lane;
      if (i < H / 8) dst[i] = v[k];
    }
  }
  // the 128-byte group-sum row: 8 lanes of 16 bytes
  if (lane < GSUM_COLS / 8)
    reinterpret_cast<uint4*>(gs_xs + (size_t)r * GSUM_COLS)[lane] =
        __ldcg(reinterpret_cast<const uint4*>(gs_xp + (size_t)t * GSUM_COLS) + lane);
}

// out[t][r] = sum_j w[t][j] * y[slot(t, j)][r] + sg[t] * ys[t][r] (+ h[t][r]), rounded to fp16 once. A thread
// takes four neighbouring columns of one token: its K slots and weights first, then the K rows' 16-byte loads,
// so that the loads are in flight together; every column adds its terms in the order above. KM >= K bounds the
// per-thread arrays.
template <int KM>
__global__ void k_chunk_combine(const float* __restrict__ y, const float* __restrict__ ys,
                                const int32_t* __restrict__ slot_of, const float* __restrict__ w,
                                const float* __restrict__ sg, const uint16_t* __restrict__ resid, int T, int H,
                                int K, uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_release();
  const int H4 = H / 4;
  const size_t n = (size_t)T * H4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), c = (int)(i % H4) * 4;
    int sl[KM];
    float wv[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < K) {
        sl[j] = __ldcg(slot_of + (size_t)t * K + j);
        wv[j] = __ldcg(w + (size_t)t * K + j);
      }
    float4 yv[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < K) yv[j] = __ldcg(reinterpret_cast<const float4*>(y + (size_t)sl[j] * H + c));
    const float4 sv = __ldcg(reinterpret_cast<const float4*>(ys + (size_t)t * H + c));
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < K) {
        a0 += wv[j] * yv[j].x;
        a1 += wv[j] * yv[j].y;
        a2 += wv[j] * yv[j].z;
        a3 += wv[j] * yv[j].w;
      }
    const float g = __ldcg(sg + t);
    a0 += g * sv.x;
    a1 += g * sv.y;
    a2 += g * sv.z;
    a3 += g * sv.w;
    if (resid) {
      const uint2 rr = __ldcg(reinterpret_cast<const uint2*>(resid + (size_t)t * H + c));
      a0 += __half2float(__ushort_as_half((uint16_t)(rr.x & 0xFFFFu)));
      a1 += __half2float(__ushort_as_half((uint16_t)(rr.x >> 16)));
      a2 += __half2float(__ushort_as_half((uint16_t)(rr.y & 0xFFFFu)));
      a3 += __half2float(__ushort_as_half((uint16_t)(rr.y >> 16)));
    }
    uint2 o;
    o.x = (uint32_t)__half_as_ushort(__float2half_rn(a0)) | ((uint32_t)__half_as_ushort(__float2half_rn(a1)) << 16);
    o.y = (uint32_t)__half_as_ushort(__float2half_rn(a2)) | ((uint32_t)__half_as_ushort(__float2half_rn(a3)) << 16);
    *reinterpret_cast<uint2*>(out + (size_t)t * H + c) = o;
  }
}

cudaError_t chunk_forward(const MoeLayout& L, const GemmLayout& G, const ChunkScratch& S, const ChunkMaps& maps,
                          int Tm, int num_sms,
                          const uint16_t* x, uint16_t* out, int T, const uint16_t* gamma, float eps,
                          int32_t* rec_ids, float* rec_w, float* rec_sg, uint32_t* status, uint64_t timeout_ns,
                          uint64_t* trace, cudaStream_t st, int* launches, int skip) {
  const int E = L.E, K = L.K, H = L.H, TW = (T + 31) / 32;
  int n = 0;
  cudaError_t e = launch_pdl(k_chunk_prologue, (T + PRO_TPC - 1) / PRO_TPC, PRO_WPT * PRO_TPC * 32, 0, st, x, gamma,
                             eps, T, H, S.xp, S.gs_xp, S.masks, E * TW);
  if (e != cudaSuccess) return e;
  ++n;
  GemmArgs ga{G, S, T, Tm, 1, status, timeout_ns, nullptr, maps, skip};
  e = chunk_gemm_launch(ga, num_sms, st);
  ga.skip = 0;
  if (e != cudaSuccess) return e;
  ++n;
  {
    auto* route = E <= 32 ? k_chunk_route<1> : E <= 64 ? k_chunk_route<2> : E <= 128 ? k_chunk_route<4>
                  : E <= 256 ? k_chunk_route<8> : k_chunk_route<16>;
    e = launch_pdl(route, (T + 7) / 8, 256, 0, st, (const float*)S.logits, router_parts(H / 64), E, K, T, S.ids,
                   S.w, S.sg, S.masks, TW, rec_ids, rec_w, rec_sg);
    if (e != cudaSuccess) return e;
  }
  ++n;
  e = launch_pdl(k_chunk_bucket, E, BUCKET_THREADS, 0, st, (const uint32_t*)S.masks, E, TW, T, K,
                 (const int32_t*)S.ids, S.slot_of, S.tok_of, S.groups, S.ctl);
  if (e != cudaSuccess) return e;
  ++n;
  e = launch_pdl(k_chunk_gather, (T * K + 7) / 8, 256, 0, st, (const uint16_t*)S.xp, (const uint16_t*)S.gs_xp,
                 (const int32_t*)S.tok_of, T * K, H, S.xs, S.gs_xs);
  if (e != cudaSuccess) return e;
  ++n;
  ga.phase = 2;
  ga.trace = trace;     // the trace holds the expert gate/up launch
  e = chunk_gemm_launch(ga, num_sms, st);
  if (e != cudaSuccess) return e;
  ++n;
  ga.phase = 3;
  ga.trace = nullptr;
  e = chunk_gemm_launch(ga, num_sms, st);
  if (e != cudaSuccess) return e;
  ++n;
  const size_t tot = (size_t)T * (H / 4);
  const int cg = (int)((tot + 255) / 256 < 65536 ? (tot + 255) / 256 : 65536);
  auto* combine = K <= 8 ? k_chunk_combine<8> : k_chunk_combine<16>;
  e = launch_pdl(combine, cg, 256, 0, st, (const float*)S.y, (const float*)S.ys, (const int32_t*)S.slot_of,
                 (const float*)S.w, (const float*)S.sg, gamma ? x : (const uint16_t*)nullptr, T, H, K, out);
  if (e != cudaSuccess) return e;
  ++n;
  if (launches) *launches = n;
  return cudaGetLastError();
}

}  // namespace moe
