// Grouped GEMMs of the prompt-chunk path on the tcgen05 tensor cores.
//
// A job is one 128-row band of a weight matrix (an expert's gate/up or down, the router, the shared expert)
// against one tile of up to 64 activation rows (tokens). For every K-tile (64 columns = one quantisation group)
// the tensor cores multiply the band's integer codes, exact in fp16, by the activations into a fresh TMEM
// accumulator D, and the tile is folded in fp32: acc += s * D + b * sum(x). The weights' affine (s, b) is thus
// applied exactly once per group instead of being rounded into fp16 weights. The B operand of the down
// projections is h split into fp16 hi + lo/4096 halves, multiplied in two MMAs into two accumulators.
//
// Persistent CTAs (one per SM) take jobs j = blockIdx.x + k * gridDim.x. Warp roles, all stepping through the
// same jobs and K-tiles and handing stages over on mbarriers:
//   warp 0     producer (one lane): a bulk copy of the K-tile's weight block (codes + pairs) and TMA tensor
//              loads of the activation rows (128-byte swizzled K-major), all on the stage's "full" barrier
//   warp 1     allocates TMEM; lane 0 issues the MMAs and commits them to the barriers that free the stage,
//              the A buffer and hand the accumulator to the fold
//   warps 2-9  dequantise, two groups of four warps taking alternate K-tiles: thread = band row, codes ->
//              exact fp16 integers in the swizzled A buffer; the threads of rows 64-127 also sum activation
//              rows 0-63 of the tile (the fold's sum(x))
//   warps 10-13 fold (thread = TMEM lane = band row) and, after the job's last K-tile, the epilogue
// Every wait is bounded; on a timeout the CTA records an error bit and every role leaves its loops.
#include <cuda_fp16.h>
#include <stdint.h>

#include "chunk.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace moe {

namespace {

enum : int { GK_ROUTER = 0, GK_SHGU = 1, GK_SHDN = 2, GK_EXGU = 3, GK_EXDN = 4 };

constexpr int GTH = 448;                // 14 warps
constexpr int NSG = 4;                  // pipeline stages
constexpr int DEPTH = 4;                // A buffers = TMEM accumulators = side buffers (K-tiles in flight
                                        // between the dequantisation and the fold)
// stage layout: weight block | B hi (64 rows x 128 B, swizzled) | B lo
constexpr int ST_W = 0, ST_BHI = 9216, ST_BLO = 17408, ST_BYTES = 25600;
constexpr int S_A = NSG * ST_BYTES;                 // DEPTH A buffers of 128 x 64 fp16 (16 KB each)
constexpr int S_SIDE = S_A + DEPTH * 16384;         // DEPTH side buffers: (s, b) of 128 rows, 64 row sums
constexpr int SIDE_BYTES = 128 * 4 + 64 * 4;
constexpr int S_XCH = S_SIDE + DEPTH * SIDE_BYTES;  // SwiGLU exchange: up values [64][65]
constexpr int S_BAR = S_XCH + 64 * 65 * 4;
constexpr int S_BYTES = S_BAR + 256;
constexpr int GEMM_SMEM = S_BYTES + 1024;           // + alignment slack
constexpr uint32_t ERR_GEMM_WAIT = 512u;

struct Job {
  int kind, m, e;
  const uint8_t* w;       // weight block of K-tile 0 of the band
  int ktiles, int8;
  int bmap, lomap;        // tensor maps of the activations and of their low halves (-1: none)
  int row0, cnt, n;       // first activation row, rows, MMA N (cnt rounded up to 16)
};

__device__ bool decode_job(const GemmArgs& g, int j, Job& jb) {
  const GemmLayout& G = g.G;
  const ChunkScratch& S = g.S;
  const int H = G.H, I = G.I, Is = G.Is, T = g.T;
  const int NTT = (T + CHUNK_NT - 1) / CHUNK_NT;
  jb.e = 0;
  jb.lomap = -1;
  auto token_tile = [&](int nt) {
    jb.row0 = nt * CHUNK_NT;
    jb.cnt = min(CHUNK_NT, T - jb.row0);
  };
  if (g.phase == 1) {
    const int MTr = G.Mr / 128, MTs = 2 * Is / 128;
    if (j < MTr * NTT) {
      jb.kind = GK_ROUTER; jb.m = j % MTr; token_tile(j / MTr);
      jb.w = G.gr + (size_t)jb.m * (H / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = H / 64;
      jb.bmap = CM_XP;
    } else {
      j -= MTr * NTT;
      if (j >= MTs * NTT) return false;
      jb.kind = GK_SHGU; jb.m = j % MTs; token_tile(j / MTs);
      jb.w = G.gsgu + (size_t)jb.m * (H / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = H / 64;
      jb.bmap = CM_XP;
    }
  } else {
    const int ngroups = S.ctl[0];
    const int MTg = 2 * I / 128, MTd = H / 128;
    const int nex = (g.phase == 2 ? MTg : MTd) * ngroups;
    if (j < nex) {
      // band-major: the row tiles of one expert for one band are consecutive jobs (they share the band's
      // weights through L2)
      const int m = j / ngroups;
      const int4 gr = S.groups[j % ngroups];
      jb.m = m; jb.e = gr.x; jb.row0 = gr.y; jb.cnt = gr.z; jb.int8 = 0;
      if (g.phase == 2) {
        jb.kind = GK_EXGU;
        jb.w = G.gegu + (size_t)gr.x * G.gegu_expert + (size_t)m * (H / 64) * GEMM_BLK4; jb.ktiles = H / 64;
        jb.bmap = CM_XS;
      } else {
        jb.kind = GK_EXDN;
        jb.w = G.gedn + (size_t)gr.x * G.gedn_expert + (size_t)m * (I / 64) * GEMM_BLK4; jb.ktiles = I / 64;
        jb.bmap = CM_HH; jb.lomap = CM_HHLO;
      }
    } else {
      j -= nex;
      if (g.phase != 2 || j >= MTd * NTT) return false;
      jb.kind = GK_SHDN; jb.m = j % MTd; token_tile(j / MTd);
      jb.w = G.gsdn + (size_t)jb.m * (Is / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = Is / 64;
      jb.bmap = CM_HS; jb.lomap = CM_HSLO;
    }
  }
  jb.n = (jb.cnt + 15) & ~15;
  return jb.cnt > 0;
}

struct Bars {
  uint64_t full[NSG], empty[NSG], a_ready[DEPTH], a_free[DEPTH], d_full[DEPTH], d_free[DEPTH];
  uint64_t fold_sync;   // the four fold warps meet here in the SwiGLU epilogue (a bounded wait)
  uint32_t tslot;
  volatile int abort;
};

// debug stamps (CTA 0, first 64 K-tiles): events 0 producer issued, 1 dequant saw the stage, 2 dequant done,
// 3 MMA issued, 4 fold saw the accumulator, 5 fold done
#define GSTAMP(ev, k) do { if (g.trace && blockIdx.x == 0 && (k) < 64) g.trace[(ev) * 64 + (k)] = clock64(); } while (0)

__device__ __forceinline__ float silu_c(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// position of unit u of an h vector in P8 order
__device__ __forceinline__ int p8u(int u) {
  const int k = u & 7;
  return (u & ~7) + (k < 4 ? 2 * k : 2 * (k - 4) + 1);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(GTH, 1) k_chunk_gemm(const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* bar = reinterpret_cast<Bars*>(smem + S_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t to = g.timeout_ns;
  auto fail = [&]() {
    atomicOr(g.status, ERR_GEMM_WAIT);
    bar->abort = 1;
  };
  // bounded wait on phase parity `ph` of `b`; false (and the CTA aborts) on a timeout or an earlier abort
  auto wait = [&](uint64_t* b, uint32_t ph) -> bool {
    if (bar->abort) return false;
    if (!mbar_wait(b, ph, to)) { fail(); return false; }
    return true;
  };

  if (tid == 0) {
    for (int s = 0; s < NSG; ++s) {
      mbar_init(&bar->full[s], 1);          // the producer's expect-tx arrival
      mbar_init(&bar->empty[s], 4 + 1);     // dequant warps (codes, pairs, sums read) + MMA commit (B read)
    }
    for (int i = 0; i < DEPTH; ++i) {
      mbar_init(&bar->a_ready[i], 4);
      mbar_init(&bar->a_free[i], 1);
      mbar_init(&bar->d_full[i], 1);
      mbar_init(&bar->d_free[i], 4);
    }
    mbar_init(&bar->fold_sync, 4);
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(&bar->tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tslot;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer (lane 0)
    if (lane == 0) {
      uint32_t gk = 0;
      bool run = true;
      for (int j = blockIdx.x; run; j += gridDim.x) {
        Job jb;
        if (!decode_job(g, j, jb)) break;
        const int blk = jb.int8 ? GEMM_BLK8 : GEMM_BLK4;
        const int box = jb.n <= 16 ? 0 : 1;
        const uint32_t bbytes = (box ? CHUNK_NT : 16) * 128;
        for (int kt = 0; kt < jb.ktiles; ++kt, ++gk) {
          const int s = gk % NSG;
          if (gk >= NSG && !wait(&bar->empty[s], ((gk / NSG) & 1u) ^ 1u)) { run = false; break; }
          uint8_t* st = smem + s * ST_BYTES;
          mbar_expect_tx(&bar->full[s], (uint32_t)blk + bbytes * (jb.lomap >= 0 ? 2u : 1u));
          bulk_g2s(st + ST_W, jb.w + (size_t)kt * blk, (uint32_t)blk, &bar->full[s]);
          tma_load_2d(st + ST_BHI, &g.maps.m[jb.bmap][box], kt * 64, jb.row0, &bar->full[s]);
          if (jb.lomap >= 0) tma_load_2d(st + ST_BLO, &g.maps.m[jb.lomap][box], kt * 64, jb.row0, &bar->full[s]);
          GSTAMP(0, gk);
        }
      }
      // drain: every copy issued must have landed before the CTA leaves
      const uint32_t cnt = gk < (uint32_t)NSG ? gk : (uint32_t)NSG;
      for (uint32_t q = gk - cnt; q < gk; ++q) mbar_wait(&bar->full[q % NSG], (q / NSG) & 1u, to);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    uint32_t gk = 0;
    bool run = true;
    for (int j = blockIdx.x; run; j += gridDim.x) {
      Job jb;
      if (!decode_job(g, j, jb)) break;
      const uint32_t idesc = umma_idesc_f16(128, jb.n);
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk) {
        const int s = gk % NSG, ab = gk % DEPTH;
        // a_ready implies that the fold of K-tile gk - DEPTH released accumulator ab (the dequantisation
        // waited for it before filling the side buffer)
        if (!wait(&bar->a_ready[ab], (gk / DEPTH) & 1u)) { run = false; break; }
        if (lane == 0) GSTAMP(6, gk);
        if (!wait(&bar->full[s], (gk / NSG) & 1u)) { run = false; break; }
        if (lane == 0) GSTAMP(7, gk);
        if (lane == 0) {
          tc_fence_after();
          uint8_t* st = smem + s * ST_BYTES;
          const uint32_t a0 = smem_u32(smem + S_A + ab * 16384);
          const uint32_t bh = smem_u32(st + ST_BHI), bl = smem_u32(st + ST_BLO);
          const uint32_t d = tmem + ab * 128;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_f16(d, umma_desc_sw128(a0 + 32 * ks), umma_desc_sw128(bh + 32 * ks), idesc, ks > 0 ? 1u : 0u);
          if (jb.lomap >= 0)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f16(d + 64, umma_desc_sw128(a0 + 32 * ks), umma_desc_sw128(bl + 32 * ks), idesc, ks > 0 ? 1u : 0u);
          umma_commit(&bar->a_free[ab]);
          umma_commit(&bar->d_full[ab]);
          umma_commit(&bar->empty[s]);
          GSTAMP(3, gk);
        }
        __syncwarp();
      }
    }
    // the last MMAs must have completed before TMEM is released
    if (lane == 0 && gk > 0) mbar_wait(&bar->d_full[(gk - 1) % DEPTH], ((gk - 1) / DEPTH) & 1u, to);
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------------------------------------ dequantise
    const int grp = (warp - 2) >> 2;          // this group takes the K-tiles gk with gk % 2 == grp
    const int r = (tid - 64) & 127;           // band row
    const __half2 k1024 = __float2half2_rn(1024.0f), k16 = __float2half2_rn(0.0625f), k64 = __float2half2_rn(-64.0f);
    uint32_t gk = 0;
    bool run = true;
    for (int j = blockIdx.x; run; j += gridDim.x) {
      Job jb;
      if (!decode_job(g, j, jb)) break;
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk) {
        if ((int)(gk & 1u) != grp) continue;
        const int s = gk % NSG, ab = gk % DEPTH;
        const uint32_t pf = ((gk / DEPTH) & 1u) ^ 1u;   // phase of K-tile gk - DEPTH
        if (!wait(&bar->full[s], (gk / NSG) & 1u) ||
            (gk >= DEPTH && (!wait(&bar->a_free[ab], pf) || !wait(&bar->d_free[ab], pf)))) {
          run = false;
          break;
        }
        if (r == 0) GSTAMP(1, gk);
        const uint8_t* st = smem + s * ST_BYTES + ST_W;
        uint8_t* A = smem + S_A + ab * 16384;
        // the fold's share of the stage goes to the side buffer, so the stage is free once the MMA has read B
        {
          uint32_t* side = reinterpret_cast<uint32_t*>(smem + S_SIDE + ab * SIDE_BYTES);
          side[r] = *reinterpret_cast<const uint32_t*>(st + 128 * (jb.int8 ? 64 : 32) + r * 4);
          const int xr = r - 64;   // activation row summed by this thread
          if (xr >= 0 && xr < jb.n) {
            // sum of activation row xr over the tile's 64 columns (swizzled 16-byte chunks); low halves / 4096
            const uint8_t* bst = smem + s * ST_BYTES;
            float sh = 0.f, sl = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t off = sw128_off(xr, c);
              const uint4 v = *reinterpret_cast<const uint4*>(bst + ST_BHI + off);
              const __half2* hv = reinterpret_cast<const __half2*>(&v);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(hv[k]);
                sh += f.x + f.y;
              }
              if (jb.lomap >= 0) {
                const uint4 u = *reinterpret_cast<const uint4*>(bst + ST_BLO + off);
                const __half2* hu = reinterpret_cast<const __half2*>(&u);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float2 f = __half22float2(hu[k]);
                  sl += f.x + f.y;
                }
              }
            }
            reinterpret_cast<float*>(side)[128 + xr] = fmaf(sl, 1.0f / 4096.0f, sh);
          }
        }
        if (jb.int8) {
          const uint8_t* codes = st + r * 64;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint2 w = *reinterpret_cast<const uint2*>(codes + c * 8);
            uint32_t v[4], o[4];
            int8_block_pairs(w.x, w.y, v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&v[k]), k1024);
              o[k] = *reinterpret_cast<const uint32_t*>(&q);
            }
            *reinterpret_cast<uint4*>(A + sw128_off(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        } else {
          const uint8_t* codes = st + r * 32;
          const uint4 w0 = *reinterpret_cast<const uint4*>(codes), w1 = *reinterpret_cast<const uint4*>(codes + 16);
          const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t v[4], o[4];
            int4_word_pairs(wd[c], v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __half2 h = *reinterpret_cast<const __half2*>(&v[k]);
              // exact codes: 1024 + q -> q; 1024 + 16 q (odd pairs) -> q
              const __half2 q = (k & 1) ? __hfma2(h, k16, k64) : __hsub2(h, k1024);
              o[k] = *reinterpret_cast<const uint32_t*>(&q);
            }
            *reinterpret_cast<uint4*>(A + sw128_off(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async_smem();   // the MMAs read A through the async proxy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar->a_ready[ab]);
          mbar_arrive(&bar->empty[s]);
        }
        if (r == 0) GSTAMP(2, gk);
      }
    }
  } else {
    // ------------------------------------------------------------------ fold + epilogue
    const int q4 = warp & 3;               // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;          // band row
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    float* xu = reinterpret_cast<float*>(smem + S_XCH);     // [64][65] up values
    const GemmLayout& G = g.G;
    const ChunkScratch& S = g.S;
    uint32_t fph = 0;
    // the four fold warps meet (bounded: a warp that has aborted makes the others time out, never hang)
    auto fold_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->fold_sync);
      const bool ok = wait(&bar->fold_sync, fph);
      fph ^= 1u;
      return ok;
    };
    uint32_t gk = 0;
    bool run = true;
    for (int j = blockIdx.x; run; j += gridDim.x) {
      Job jb;
      if (!decode_job(g, j, jb)) break;
      float acc[CHUNK_NT];
#pragma unroll
      for (int i = 0; i < CHUNK_NT; ++i) acc[i] = 0.f;
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk) {
        const int ab = gk % DEPTH;
        // the dequantisation released the side buffer with a_ready (already complete once d_full is)
        if (!wait(&bar->d_full[ab], (gk / DEPTH) & 1u) || !wait(&bar->a_ready[ab], (gk / DEPTH) & 1u)) {
          run = false;
          break;
        }
        tc_fence_after();
        if (r == 0) GSTAMP(4, gk);
        const uint32_t* side = reinterpret_cast<const uint32_t*>(smem + S_SIDE + ab * SIDE_BYTES);
        const float2 sb = h2f(side[r]);
        const float* xs = reinterpret_cast<const float*>(side + 128);
        const uint32_t d = trow + ab * 128;
#pragma unroll
        for (int c0 = 0; c0 < CHUNK_NT; c0 += 16) {
          if (c0 < jb.n) {
            uint32_t vh[16], vl[16];
            tmem_ld16_nowait(d + c0, vh);
            if (jb.lomap >= 0) tmem_ld16_nowait(d + 64 + c0, vl);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float dv = __uint_as_float(vh[i]);
              if (jb.lomap >= 0) dv = fmaf(__uint_as_float(vl[i]), 1.0f / 4096.0f, dv);
              acc[c0 + i] = fmaf(sb.x, dv, fmaf(sb.y, xs[c0 + i], acc[c0 + i]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->d_free[ab]);
        if (r == 0) GSTAMP(5, gk);
      }
      if (!run) break;
      // ---- epilogue: thread = band row r, columns = the tile's tokens
      if (jb.kind == GK_ROUTER) {
        const int er = jb.m * 128 + r;
        if (er <= G.E)
#pragma unroll
          for (int i = 0; i < CHUNK_NT; ++i)
            if (i < jb.cnt) S.logits[(size_t)(jb.row0 + i) * (G.E + 1) + er] = acc[i];
      } else if (jb.kind == GK_SHDN || jb.kind == GK_EXDN) {
        float* dst = jb.kind == GK_SHDN ? S.ys : S.y;
#pragma unroll
        for (int i = 0; i < CHUNK_NT; ++i)
          if (i < jb.cnt) dst[(size_t)(jb.row0 + i) * G.H + jb.m * 128 + r] = acc[i];
      } else {
        // SwiGLU: rows 0-63 are gate units 64m.., rows 64-127 the matching up units. h = silu(g) * u is split
        // into fp16 hi + lo/4096 halves, the down projection's B operand.
        const bool sh = jb.kind == GK_SHGU;
        const int kd = sh ? G.Is : G.I;
        uint16_t* dhi = sh ? S.hs : S.hh;
        uint16_t* dlo = sh ? S.hs_lo : S.hh_lo;
        if (r >= 64)
#pragma unroll
          for (int i = 0; i < CHUNK_NT; ++i) xu[(r - 64) * 65 + i] = acc[i];
        if (!fold_sync()) break;
        if (r < 64) {
          const int pos = p8u(jb.m * 64 + r);
#pragma unroll
          for (int i = 0; i < CHUNK_NT; ++i) {
            if (i < jb.cnt) {
              const float h = silu_c(acc[i]) * xu[r * 65 + i];
              const __half hh = __float2half_rn(h);
              const __half hl = __float2half_rn((h - __half2float(hh)) * 4096.0f);
              const size_t o = (size_t)(jb.row0 + i) * kd + pos;
              dhi[o] = __half_as_ushort(hh);
              dlo[o] = __half_as_ushort(hl);
            }
          }
        }
        if (!fold_sync()) break;   // the exchange buffer is free for the next job
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t chunk_gemm_launch(const GemmArgs& g, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_chunk_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k_chunk_gemm<<<grid, GTH, GEMM_SMEM, st>>>(g);
  return cudaGetLastError();
}

}  // namespace moe
