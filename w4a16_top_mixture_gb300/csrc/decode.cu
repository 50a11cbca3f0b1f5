// Fused decode kernel of the W4A16 routed-MoE block (T <= 16 tokens): one cooperative, persistent launch with
// one CTA per SM.
//
// Roles inside a CTA: warp 0 is the producer (one lane issues 1-D bulk copies of contiguous weight ranges
// into a ring of shared-memory stages, each guarded by a "full" and an "empty" mbarrier); warps 1..16 are
// consumers. Work a CTA owns, in stream order:
//   A1  its share of the router rows (int8)           -> logits to global, then a grid-wide arrival count
//   R   routing: every CTA waits for all logits and computes softmax -> top-k -> renormalise for every token
//       itself (identical arithmetic everywhere), then buckets tokens by expert
//   A2  its share of the shared-expert gate/up units   -> hs = silu(g)*u to global, arrival count
//   B   its share of the routed units: all (active expert, intermediate unit) pairs split evenly across the
//       grid. For each unit: h = silu(Wg x)*(Wu x) per routed token, then that unit's column of the down
//       matrix times h, accumulated per output row into a weighted partial sum per (segment, token)
//   C   its share of the shared-down output rows (needs all hs: waits on the hs arrival count)
//   D   after a grid-wide count of finished partials: for its output rows, out = sum of the partials in a
//       fixed order + sigmoid(g) * shared row (+ residual), rounded to fp16 once
// Every grid-wide or mbarrier wait is bounded by a timeout; a timeout records an error bit and the CTA
// drains its in-flight copies and leaves, so no wait can hang the GPU.
#include <cuda_fp16.h>
#include <stdint.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int NCW = DEC_NCW;
constexpr int CT = NCW * 32;   // consumer threads
constexpr int BAR_C = 1;       // named barrier of all consumer warps
constexpr int BAR_A = 2;       // the shared-expert team
constexpr int BAR_R = 3;       // the routing team
constexpr uint32_t FULL = 0xFFFFFFFFu;

constexpr size_t c_align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Compile-time block shape: every width, stride and loop bound of the decode kernel is a constant, which keeps
// its machine code small (the kernel's executed code must stay resident in the SM instruction cache).
template <int H_, int E_, int K_, int I_, int Is_>
struct Shape {
  static constexpr int H = H_, E = E_, K = K_, I = I_, Is = Is_;
  static constexpr int GB = H / 64, GI = I / 64, GS = Is / 64;
  static constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  static constexpr size_t RR = c_align16((size_t)H + (size_t)GB * 4);
  static constexpr size_t SU = c_align16(2 * (size_t)H + 2 * (size_t)GB * 4);
  static constexpr size_t SDR = c_align16((size_t)Is + (size_t)GS * 4);
  static constexpr size_t EU = c_align16((size_t)H + 2 * (size_t)GB * 4);
  static constexpr size_t DSB = (size_t)H * 4;
  static constexpr size_t DCB = (size_t)H / 2;
  static constexpr size_t DB = DSB + 64 * DCB;
  static constexpr size_t exgu_expert = (size_t)I * EU;
  static constexpr size_t exdn_expert = (size_t)GI * DB;
};
using ShapeProd = Shape<2048, 256, 8, 512, 512>;
using ShapeTiny = Shape<512, 32, 4, 128, 128>;

struct Ctl {
  uint64_t full[DEC_MAXNS];
  uint64_t empty[DEC_MAXNS];
  uint64_t route_ready;
  volatile int abort;
  int U;
  int nseg;
  int issued;
  int seg_a[DEC_MAXSEG], seg_e[DEC_MAXSEG], seg_u0[DEC_MAXSEG], seg_u1[DEC_MAXSEG], seg_n[DEC_MAXSEG];
  uint8_t seg_tok[DEC_MAXSEG][DEC_TMAX];
  float seg_w[DEC_MAXSEG][DEC_TMAX];
  int ids[DEC_TMAX][16];
  float wts[DEC_TMAX][16];
  float sg[DEC_TMAX];
  float rn[DEC_TMAX];
  uint32_t emask[512];
  uint16_t act_e[512];
  uint32_t act_mask[512];
  int warp_tot[NCW];
  uint16_t tab_a0[DEC_MAXGRID];   // per CTA: first active-expert index of its unit range
  uint8_t tab_n[DEC_MAXGRID];     // per CTA: number of segments
  int nslot[DEC_TMAX];            // per token: number of partial-sum slots holding it
  uint16_t slot[DEC_TMAX][2 * DEC_MAXGRID];   // per token: the slots, in (CTA, segment) order
};
constexpr int CTL_BYTES = (sizeof(Ctl) + 127) & ~127;

struct Smem {   // byte offsets of the dynamic shared-memory regions
  int xh, xs, hss, hseg, shs, ring;
};

// xh: x as fp16 [T][P][4 blocks][LW lanes] uint4 (the 8 columns of a block in pair order 0 4 1 5 2 6 3 7);
// xs: per (token, 32-column chunk) the sums of x over the chunk's "low" and "high" pair columns;
// hseg: phase B's h, and before phase B the shared expert's hs [T][Is]; hss: 16-column sums of hs;
// shs: this CTA's shared-down rows; ring: the weight stages.
template <class LT>
__host__ __device__ inline Smem smem_map(const LT& L, int T, int grid, int hseg_floats) {
  Smem m;
  int o = CTL_BYTES;
  m.xh = o;   o += (T * L.H * 2 + 127) & ~127;
  m.xs = o;   o += (T * L.NCH * 8 + 127) & ~127;
  m.hss = o;  o += (T * (L.Is / 16) * 4 + 127) & ~127;
  m.hseg = o;
  {
    int hx = hseg_floats > T * L.Is ? hseg_floats : T * L.Is;
    o += (hx * 4 + 127) & ~127;
  }
  int rpc = (L.H + grid - 1) / grid;
  m.shs = o;  o += (T * rpc * 4 + 127) & ~127;
  m.ring = o;
  return m;
}

__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)(((unsigned)n * (unsigned)c) / (unsigned)G); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}


__device__ __forceinline__ void stamp(const DecodeArgs& a, int slot) {
  if (a.trace) a.trace[blockIdx.x * 32 + slot] = globaltimer();
}
// per-warp stamps (lane 0): trace[grid*32 + (cta*16 + warp)*4 + k]
__device__ __forceinline__ void wstamp(const DecodeArgs& a, int cw, int k) {
  if (a.trace && (threadIdx.x & 31) == 0) a.trace[gridDim.x * 32 + (blockIdx.x * 16 + cw) * 4 + k] = globaltimer();
}

__device__ __forceinline__ void set_error(const DecodeArgs& a, Ctl* ctl, uint32_t bit) {
  atomicOr(a.status, bit);
  ctl->abort = 1;
}

template <int NR, int TK>
struct DotR {
  float v[TK][NR];
};

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Dot products of NR rows (a warp's work item) with up to TK tokens. INT8 = false: int4 rows in canonical
// packing; INT8 = true: permuted int8 rows. Lane l covers the 32-column chunks c = l + LW*p. Every code enters
// as the exact fp16 value 1024 + q (or 1024 + 16q) and is multiplied by the fp16 activation in an
// f16 x f16 -> f32 fused multiply-add; the 1024 offsets are removed once per chunk with the chunk's x sums.
// Returns the warp-reduced sums v[tt][r] = sum_c (s_g(c) * dot_c + b_g(c) * xsum_c) in every lane. Kept out of
// line: one copy per (NR, INT8) keeps the kernel's executed code within the SM instruction cache.
template <int H, int NR, int TK, bool INT8>
__device__ __noinline__ DotR<NR, TK> dot_rows(const uint8_t* r0, const uint8_t* r1, const uint8_t* r2,
                                              const uint8_t* r3, const uint8_t* s0, const uint8_t* s1,
                                              const uint8_t* s2, const uint8_t* s3, int nvalid,
                                              const uint4* __restrict__ xh, const float2* __restrict__ xs, int ta,
                                              int tb, int nt) {
  constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  const int lane = threadIdx.x & 31;
  const uint8_t* rp[4] = {r0, r1, r2, r3};
  const uint8_t* sp[4] = {s0, s1, s2, s3};
  int tix[TK];
  tix[0] = ta;
  if (TK > 1) tix[TK - 1] = tb;
  DotR<NR, TK> out;
#pragma unroll
  for (int tt = 0; tt < TK; ++tt)
#pragma unroll
    for (int r = 0; r < NR; ++r) out.v[tt][r] = 0.f;
  if (lane < LW) {
#pragma unroll 1
    for (int p = 0; p < P; ++p) {
      const int c = lane + LW * p;
      float lo[TK][NR], hi[TK][NR];
#pragma unroll
      for (int tt = 0; tt < TK; ++tt)
#pragma unroll
        for (int r = 0; r < NR; ++r) lo[tt][r] = hi[tt][r] = 0.f;
      uint4 ca[NR], cb[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (INT8) {
          ca[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + ((p * 2) * LW + lane) * 16) : make_uint4(0, 0, 0, 0);
          cb[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + ((p * 2 + 1) * LW + lane) * 16) : make_uint4(0, 0, 0, 0);
        } else {
          ca[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rp[r] + c * 16) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // 8-column block j of the chunk
        uint4 xv[TK];
#pragma unroll
        for (int tt = 0; tt < TK; ++tt)
          xv[tt] = tt < nt ? xh[((tix[tt] * P + p) * 4 + j) * LW + lane] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          uint32_t v[4];
          if (INT8) {
            const uint4& q4 = j < 2 ? ca[r] : cb[r];
            int8_block_pairs((j & 1) ? q4.z : q4.x, (j & 1) ? q4.w : q4.y, v);
          } else {
            int4_word_pairs(j == 0 ? ca[r].x : j == 1 ? ca[r].y : j == 2 ? ca[r].z : ca[r].w, v);
          }
#pragma unroll
          for (int tt = 0; tt < TK; ++tt) {
            lo[tt][r] = fmix_lo(v[0], xv[tt].x, lo[tt][r]);
            lo[tt][r] = fmix_hi(v[0], xv[tt].x, lo[tt][r]);
            hi[tt][r] = fmix_lo(v[1], xv[tt].y, hi[tt][r]);
            hi[tt][r] = fmix_hi(v[1], xv[tt].y, hi[tt][r]);
            lo[tt][r] = fmix_lo(v[2], xv[tt].z, lo[tt][r]);
            lo[tt][r] = fmix_hi(v[2], xv[tt].z, lo[tt][r]);
            hi[tt][r] = fmix_lo(v[3], xv[tt].w, hi[tt][r]);
            hi[tt][r] = fmix_hi(v[3], xv[tt].w, hi[tt][r]);
          }
        }
      }
      // remove the 1024 offsets, then the group's affine: s * sum(q x) + b * sum(x)
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < nvalid) {
          const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(sp[r] + (c >> 1) * 4));
#pragma unroll
          for (int tt = 0; tt < TK; ++tt) {
            const float2 X = tt < nt ? xs[(tix[tt] * P + p) * LW + lane] : make_float2(0.f, 0.f);
            const float d = (lo[tt][r] - 1024.0f * X.x) + (hi[tt][r] - 1024.0f * X.y) * (INT8 ? 1.0f : 0.0625f);
            out.v[tt][r] += sb.x * d + sb.y * (X.x + X.y);
          }
        }
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < TK; ++tt)
#pragma unroll
    for (int r = 0; r < NR; ++r) out.v[tt][r] = warp_sum(out.v[tt][r]);
  return out;
}

// Top-k of one token's expert logits held by a warp. Lane l holds experts l*EPL .. l*EPL+EPL-1 (a lower lane
// means lower indices) as order-preserving integer keys. Each of the k rounds takes the warp maximum of the lane
// maxima (the lowest lane winning ties; within a lane the lowest index), and only the winning lane recomputes
// its maximum. Lane j < k returns the j-th largest (index, logit).
// Once the k experts are known, lane j asks L2 to prefetch this CTA's 1/G slice of the j-th one's weights
// (pf_gu / pf_dn: the expert blocks, pf_gu_sz / pf_dn_sz bytes each): the grid as a whole starts pulling the
// selected experts into L2 while the bucketing runs, ahead of the weight copies that follow it.
template <int EPL>
__device__ __noinline__ void warp_topk(const float* __restrict__ lg, int E, int K, int lane, int& my_idx,
                                       float& my_logit, const uint8_t* pf_gu, size_t pf_gu_sz,
                                       const uint8_t* pf_dn, size_t pf_dn_sz) {
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane * EPL + i;
    const uint32_t b = e < E ? __float_as_uint(__ldcg(lg + e)) : 0u;
    key[i] = e < E ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
  }
  uint32_t best = key[0];
  int bi = 0;
#pragma unroll
  for (int i = 1; i < EPL; ++i)
    if (key[i] > best) { best = key[i]; bi = i; }
  my_idx = -1;
  uint32_t my_key = 0;
  const int G = gridDim.x, c = blockIdx.x;
  const size_t gu0 = ((pf_gu_sz * c / G) & ~(size_t)15), gu1 = ((pf_gu_sz * (c + 1) / G) & ~(size_t)15);
  const size_t dn0 = ((pf_dn_sz * c / G) & ~(size_t)15), dn1 = ((pf_dn_sz * (c + 1) / G) & ~(size_t)15);
#pragma unroll 1
  for (int j = 0; j < K; ++j) {
    const uint32_t m = __reduce_max_sync(FULL, best);
    const int win = __ffs(__ballot_sync(FULL, best == m)) - 1;
    const int sel = __shfl_sync(FULL, lane * EPL + bi, win);
    if (lane == j) { my_idx = sel; my_key = m; }
    if (lane == win) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == bi) key[i] = 0u;
      best = key[0];
      bi = 0;
#pragma unroll
      for (int i = 1; i < EPL; ++i)
        if (key[i] > best) { best = key[i]; bi = i; }
    }
  }
  // lane j < k starts the L2 prefetch of this CTA's slice of the j-th selected expert
  if (lane < K && pf_gu) {
    if (gu1 > gu0) prefetch_l2(pf_gu + (size_t)my_idx * pf_gu_sz + gu0, (uint32_t)(gu1 - gu0));
    if (dn1 > dn0) prefetch_l2(pf_dn + (size_t)my_idx * pf_dn_sz + dn0, (uint32_t)(dn1 - dn0));
  }
  const uint32_t b = (my_key & 0x80000000u) ? (my_key & 0x7FFFFFFFu) : ~my_key;
  my_logit = __uint_as_float(b);
}

template <class SH, int TK>
__global__ void __launch_bounds__(DEC_THREADS, 1) k_decode(DecodeArgs a, int NS, int SS, int hseg_floats) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr SH L{};
  constexpr int H = SH::H, NCH = SH::NCH, LW = SH::LW, P = SH::P;
  constexpr int E = SH::E, K = SH::K, I = SH::I, Is = SH::Is;
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  const Smem sm = smem_map(L, T, G, hseg_floats);
  uint4* xh = reinterpret_cast<uint4*>(smem + sm.xh);
  float2* xs = reinterpret_cast<float2*>(smem + sm.xs);
  float* hss = reinterpret_cast<float*>(smem + sm.hss);
  float* hseg = reinterpret_cast<float*>(smem + sm.hseg);
  float* hsn = hseg;   // shared-expert hs [T][Is], natural order, used before phase B
  float* shs = reinterpret_cast<float*>(smem + sm.shs);
  uint8_t* ring = smem + sm.ring;

  // per-CTA static ranges
  const int ra = range_lo(E + 1, cta, G), rb = range_lo(E + 1, cta + 1, G);       // router rows
  const int sa = range_lo(Is, cta, G), sbn = range_lo(Is, cta + 1, G);           // shared units
  const int r0 = range_lo(H, cta, G), r1 = range_lo(H, cta + 1, G);             // output rows
  const int RPI = SS / (int)L.RR;                 // router rows per item
  const int SPI = (SS / (int)L.SU) & ~1;          // shared units per item (even)
  const int UPI = (SS / (int)L.EU) & ~1;          // expert units per item (even)
  const int DPI = SS / (int)L.DCB;                // down columns per item
  const int SDPI = SS / (int)L.SDR;               // shared-down rows per item

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], NCW);
    }
    mbar_init(&ctl->route_ready, 1);
    ctl->abort = 0;
    ctl->issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp(a, 0);

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int n = 0, ps = 0;      // items issued, ring stage of the next one
      uint32_t pph = 0;       // wrap parity of the ring
      const uint64_t pol = policy_evict_first();
      auto issue = [&](const uint8_t* src, uint32_t bytes) -> bool {
        if (ctl->abort) return false;
        if (n >= NS && !mbar_wait(&ctl->empty[ps], pph ^ 1u, a.timeout_ns)) {
          set_error(a, ctl, ERR_WAIT_EMPTY);
          return false;
        }
        mbar_expect_tx(&ctl->full[ps], bytes);
        bulk_g2s_hint(ring + (size_t)ps * SS, src, bytes, &ctl->full[ps], pol);
        ++n;
        if (++ps == NS) { ps = 0; pph ^= 1u; }
        return true;
      };
      bool ok = true;
#pragma unroll 1
      for (int r = ra; ok && r < rb; r += RPI)
        ok = issue(a.router + (size_t)r * L.RR, (uint32_t)(min(RPI, rb - r) * L.RR));
#pragma unroll 1
      for (int u = sa; ok && u < sbn; u += SPI)
        ok = issue(a.sh_gu + (size_t)u * L.SU, (uint32_t)(min(SPI, sbn - u) * L.SU));
#pragma unroll 1
      for (int r = r0; ok && r < r1; r += SDPI)
        ok = issue(a.sh_dn + (size_t)r * L.SDR, (uint32_t)(min(SDPI, r1 - r) * L.SDR));
      stamp(a, 16);
      if (ok && !mbar_wait(&ctl->route_ready, 0, a.timeout_ns * 4)) {
        set_error(a, ctl, ERR_WAIT_ROUTE);
        ok = false;
      }
      if (ok && ctl->abort) ok = false;
      stamp(a, 17);
      const int nseg = ok ? ctl->nseg : 0;
#pragma unroll 1
      for (int sgi = 0; ok && sgi < nseg; ++sgi) {
        const int e = ctl->seg_e[sgi], u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi];
        const uint8_t* gu = a.ex_gu + (size_t)e * L.exgu_expert;
#pragma unroll 1
        for (int u = u0; ok && u < u1; u += UPI)
          ok = issue(gu + (size_t)u * L.EU, (uint32_t)(min(UPI, u1 - u) * L.EU));
        const uint8_t* dn = a.ex_dn + (size_t)e * L.exdn_expert;
#pragma unroll 1
        for (int g = u0 / 64; ok && g * 64 < u1; ++g) {
          const uint8_t* blk = dn + (size_t)g * L.DB;
          ok = issue(blk, (uint32_t)L.DSB);
          const int ga = max(u0, g * 64), gb = min(u1, g * 64 + 64);
#pragma unroll 1
          for (int u = ga; ok && u < gb; u += DPI)
            ok = issue(blk + L.DSB + (size_t)(u - g * 64) * L.DCB, (uint32_t)(min(DPI, gb - u) * L.DCB));
        }
      }
      stamp(a, 18);
      // drain: every issued copy must have landed before the CTA may leave
      {
        // the last min(n, NS) issued items, oldest first: walk back from the next stage
        const int cnt = min(n, NS);
        int s = ps - cnt;
        uint32_t ph = pph;
        if (s < 0) { s += NS; ph ^= 1u; }
#pragma unroll 1
        for (int m = 0; m < cnt; ++m) {
          if (!mbar_wait(&ctl->full[s], ph, a.timeout_ns)) atomicOr(a.status, ERR_WAIT_FULL);
          if (++s == NS) { s = 0; ph ^= 1u; }
        }
      }
      stamp(a, 19);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    int cs = 0;            // ring stage of the next item, mirrors the producer's order
    uint32_t cph = 0;      // its phase parity
    auto acquire = [&]() -> const uint8_t* {
      if (!ctl->abort && !mbar_wait(&ctl->full[cs], cph, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_FULL);
      return ring + (size_t)cs * SS;
    };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[cs]);
      if (++cs == NS) { cs = 0; cph ^= 1u; }
    };

    // ---- x prologue: (RMSNorm ->) fp16 activations in pair order, plus per-chunk pair-column sums; one
    // (token, 32-column chunk) item per consumer thread
    if (a.gamma) {
#pragma unroll 1
      for (int t = cw; t < T; t += NCW) {
        const uint16_t* xr = a.x + (size_t)t * H;
        float ss = 0.f;
#pragma unroll 1
        for (int i = lane * 8; i < H; i += 256) {
          const uint4 raw = *reinterpret_cast<const uint4*>(xr + i);
          const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(hv[k]);
            ss += f.x * f.x + f.y * f.y;
          }
        }
        ss = warp_sum(ss);
        if (lane == 0) ctl->rn[t] = 1.0f / sqrtf(ss / (float)H + a.eps);
      }
      named_bar(BAR_C, CT);
    }
#pragma unroll 1
    for (int item = ctid; item < T * NCH; item += CT) {
      const int t = item / NCH, c = item % NCH, l = c % LW, p = c / LW;
      const uint16_t* xr = a.x + (size_t)t * H + c * 32;
      uint4 raw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) raw[j] = *reinterpret_cast<const uint4*>(xr + j * 8);
      const float rn = a.gamma ? ctl->rn[t] : 1.f;
      float xl = 0.f, xhs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half h8[8];
        *reinterpret_cast<uint4*>(h8) = raw[j];
        if (a.gamma) {
          const uint4 graw = *reinterpret_cast<const uint4*>(a.gamma + c * 32 + j * 8);
          const __half* g8 = reinterpret_cast<const __half*>(&graw);
#pragma unroll
          for (int k = 0; k < 8; ++k) h8[k] = __float2half_rn(__half2float(h8[k]) * rn * __half2float(g8[k]));
        }
        // pair order (0,4) (1,5) (2,6) (3,7); "low" columns 0 4 2 6, "high" columns 1 5 3 7
        uint4 o;
        o.x = (uint32_t)__half_as_ushort(h8[0]) | ((uint32_t)__half_as_ushort(h8[4]) << 16);
        o.y = (uint32_t)__half_as_ushort(h8[1]) | ((uint32_t)__half_as_ushort(h8[5]) << 16);
        o.z = (uint32_t)__half_as_ushort(h8[2]) | ((uint32_t)__half_as_ushort(h8[6]) << 16);
        o.w = (uint32_t)__half_as_ushort(h8[3]) | ((uint32_t)__half_as_ushort(h8[7]) << 16);
        xh[((t * P + p) * 4 + j) * LW + l] = o;
        xl += (__half2float(h8[0]) + __half2float(h8[4])) + (__half2float(h8[2]) + __half2float(h8[6]));
        xhs += (__half2float(h8[1]) + __half2float(h8[5])) + (__half2float(h8[3]) + __half2float(h8[7]));
      }
      xs[(t * P + p) * LW + l] = make_float2(xl, xhs);
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 1);

    // ---- A1: router rows -> logits (a row per warp)
    for (int r = ra; r < rb; r += RPI) {
      const int nr = min(RPI, rb - r);
      const uint8_t* st = acquire();
      if (!ctl->abort) {
        const int rbase = r - ra;
#pragma unroll 1
        for (int rr = (cw - rbase % NCW + NCW) % NCW; rr < nr; rr += NCW) {
          const uint8_t* b0 = st + (size_t)rr * L.RR;
          for (int tc = 0; tc < T; tc += TK) {
            const int nt = min(TK, T - tc);
            const DotR<1, TK> d = dot_rows<H, 1, TK, true>(b0, b0, b0, b0, b0 + H, b0 + H, b0 + H, b0 + H, 1, xh, xs,
                                                           tc, tc + TK - 1, nt);
            if (lane == 0)
#pragma unroll
              for (int tt = 0; tt < TK; ++tt)
                if (tt < nt) a.logits[(size_t)(tc + tt) * (E + 1) + r + rr] = d.v[tt][0];
          }
        }
      }
      release();
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) {
      stamp(a, 2);
      if (!(a.skip_arrive && cta == 0)) {
        __threadfence();
        atomicAdd(&a.counters[0], 1u);
      }
    }

    // The warps split in two teams: RW routing warps wait for every CTA's logits and route, while the other AW
    // warps compute this CTA's shared-expert gate/up units; both join again before the shared down rows.
    const int RW = T < 8 ? T : 8, AW = NCW - RW;
    if (cw < AW) {
      // ---- A2: shared-expert gate/up units, a pair per warp
#pragma unroll 1
      for (int u = sa; u < sbn; u += SPI) {
        const int nu = min(SPI, sbn - u);
        const uint8_t* st = acquire();
        if (!ctl->abort) {
          const int pbase = (u - sa) >> 1;
#pragma unroll 1
          for (int pr = (cw - pbase % AW + AW) % AW; pr * 2 < nu; pr += AW) {
            const uint8_t* ub = st + (size_t)(2 * pr) * L.SU;
            const int nvalid = (2 * pr + 1 < nu) ? 4 : 2;
            const int i0 = u + 2 * pr;
#pragma unroll 1
            for (int tc = 0; tc < T; tc += TK) {
              const int nt = min(TK, T - tc);
              const DotR<4, TK> d = dot_rows<H, 4, TK, true>(ub, ub + H, ub + L.SU, ub + L.SU + H, ub + 2 * H,
                                                             ub + 2 * H + L.GB * 4, ub + L.SU + 2 * H,
                                                             ub + L.SU + 2 * H + L.GB * 4, nvalid, xh, xs, tc,
                                                             tc + TK - 1, nt);
              if (lane < 2 * TK) {
                const int tt = lane >> 1, k = lane & 1;
                float g = 0.f, up = 0.f;
#pragma unroll
                for (int q = 0; q < TK; ++q)
                  if (q == tt) { g = k ? d.v[q][2] : d.v[q][0]; up = k ? d.v[q][3] : d.v[q][1]; }
                if (tt < nt && 2 * k < nvalid) a.hs[(size_t)(tc + tt) * Is + i0 + k] = silu_fast(g) * up;
              }
            }
          }
        }
        release();
      }
      named_bar(BAR_A, AW * 32);
      if (ctid == 0) {
        __threadfence();
        atomicAdd(&a.counters[1], 1u);
        stamp(a, 6);
      }
    } else {
      const int rt = cw - AW, rtid = ctid - AW * 32, NT = RW * 32;
      // this team does not read the shared-expert items: it only counts itself out of their stages
#pragma unroll 1
      for (int u = sa; u < sbn; u += SPI) release();
      // ---- R: routing (every CTA, every token)
      if (rtid == 0 && !ctl->abort && !spin_geq(&a.counters[0], (uint32_t)G, a.timeout_ns))
        set_error(a, ctl, ERR_WAIT_LOGITS);
      if (rtid == 0) stamp(a, 3);
      named_bar(BAR_R, NT);
      if (!ctl->abort) {
#pragma unroll 1
        for (int t = rt; t < T; t += RW) {
          const float* lg = a.logits + (size_t)t * (E + 1);
          int my_idx;
          float my_logit;
          warp_topk<(E + 31) / 32>(lg, E, K, lane, my_idx, my_logit, a.ex_gu, L.exgu_expert, a.ex_dn,
                                   L.exdn_expert);
          const float mx = __shfl_sync(FULL, my_logit, 0);
          const float ex = lane < K ? __expf(my_logit - mx) : 0.f;
          const float Z = warp_sum(ex);
          int rank = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int oi = __shfl_sync(FULL, my_idx, i);
            rank += (i < K && oi < my_idx) ? 1 : 0;
          }
          if (lane < K) {
            ctl->ids[t][rank] = my_idx;
            ctl->wts[t][rank] = __fdividef(ex, Z);
          }
          if (lane == 0) ctl->sg[t] = __frcp_rn(1.0f + __expf(-__ldcg(lg + E)));
        }
      }
      named_bar(BAR_R, NT);
      if (rtid == 0) stamp(a, 4);
      // bucketing: token masks per expert, active experts in ascending order
      if (T == 1) {
        if (rtid < K) {
          ctl->act_e[rtid] = (uint16_t)ctl->ids[0][rtid];
          ctl->act_mask[rtid] = 1u;
        }
        if (rtid == 0) ctl->U = ctl->abort ? 0 : K;
      } else {
#pragma unroll 1
        for (int e = rtid; e < E; e += NT) ctl->emask[e] = 0u;
        named_bar(BAR_R, NT);
        if (!ctl->abort)
#pragma unroll 1
          for (int p = rtid; p < T * K; p += NT) atomicOr(&ctl->emask[ctl->ids[p / K][p % K]], 1u << (p / K));
        named_bar(BAR_R, NT);
        const int EPT = (E + NT - 1) / NT;
        int cnt = 0;
#pragma unroll 1
        for (int q = 0; q < EPT; ++q) {
          const int e = rtid * EPT + q;
          cnt += (e < E && ctl->emask[e] != 0u) ? 1 : 0;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += v;
        }
        if (lane == 31) ctl->warp_tot[rt] = incl;
        named_bar(BAR_R, NT);
        int base = 0;
#pragma unroll 1
        for (int w = 0; w < rt; ++w) base += ctl->warp_tot[w];
        int pos = base + incl - cnt;
#pragma unroll 1
        for (int q = 0; q < EPT; ++q) {
          const int e = rtid * EPT + q;
          const uint32_t msk = e < E ? ctl->emask[e] : 0u;
          if (msk != 0u) {
            ctl->act_e[pos] = (uint16_t)e;
            ctl->act_mask[pos] = msk;
            ++pos;
          }
        }
        if (rtid == NT - 1) ctl->U = base + incl;
      }
      named_bar(BAR_R, NT);
      const int U = ctl->U;
      const int N = U * I;
      if (rtid == 0) {
        const int lo = range_lo(N, cta, G), hi = range_lo(N, cta + 1, G);
        int nseg = 0;
#pragma unroll 1
        for (int aa = lo / I; aa * I < hi && lo < hi; ++aa) {
          if (nseg == DEC_MAXSEG) { set_error(a, ctl, ERR_SEGMENTS); break; }
          const int e = ctl->act_e[aa];
          const uint32_t msk = ctl->act_mask[aa];
          ctl->seg_e[nseg] = e;
          ctl->seg_u0[nseg] = max(lo, aa * I) - aa * I;
          ctl->seg_u1[nseg] = min(hi, (aa + 1) * I) - aa * I;
          int n = 0;
#pragma unroll 1
          for (int t = 0; t < T; ++t) {
            if (msk & (1u << t)) {
              ctl->seg_tok[nseg][n] = (uint8_t)t;
              float wv = 0.f;
#pragma unroll 1
              for (int j = 0; j < K; ++j)
                if (ctl->ids[t][j] == e) wv = ctl->wts[t][j];
              ctl->seg_w[nseg][n] = wv;
              ++n;
            }
          }
          ctl->seg_n[nseg] = n;
          const int units = ctl->seg_u1[nseg] - ctl->seg_u0[nseg];
          if (units * n > hseg_floats) set_error(a, ctl, ERR_HSEG);
          ++nseg;
        }
        ctl->nseg = ctl->abort ? 0 : nseg;
        mbar_arrive(&ctl->route_ready);
        stamp(a, 5);
      }
      // off the critical path: every CTA's segment table and, per token, the list of partial-sum slots that
      // hold it (final reduction)
#pragma unroll 1
      for (int c = rtid; c < G; c += NT) {
        const int lo = range_lo(N, c, G), hi = range_lo(N, c + 1, G);
        ctl->tab_a0[c] = (uint16_t)(lo / I);
        ctl->tab_n[c] = (uint8_t)(lo < hi ? (hi - 1) / I - lo / I + 1 : 0);
      }

      if (cta == 0 && a.rec_ids) {
#pragma unroll 1
        for (int p = rtid; p < T * K; p += NT) {
          a.rec_ids[p] = ctl->ids[p / K][p % K];
          a.rec_w[p] = ctl->wts[p / K][p % K];
        }
#pragma unroll 1
        for (int t = rtid; t < T; t += NT) a.rec_sg[t] = ctl->sg[t];
      }
    }
    named_bar(BAR_C, CT);

    // ---- C: shared down rows (every CTA's hs; the routed weights are in flight meanwhile)
    if (ctid == 0 && !ctl->abort && !spin_geq(&a.counters[1], (uint32_t)G, a.timeout_ns))
      set_error(a, ctl, ERR_WAIT_HS);
    named_bar(BAR_C, CT);
    if (!ctl->abort)
#pragma unroll 1
      for (int i = ctid; i < T * Is / 4; i += CT)
        reinterpret_cast<float4*>(hsn)[i] = __ldcg(reinterpret_cast<const float4*>(a.hs) + i);
    named_bar(BAR_C, CT);
    if (!ctl->abort)
#pragma unroll 1
      for (int i = ctid; i < T * (Is / 16); i += CT) {
        const float4* src = reinterpret_cast<const float4*>(hsn + (size_t)i * 16);
        const float4 p0 = src[0], p1 = src[1], p2 = src[2], p3 = src[3];
        hss[i] = ((p0.x + p0.y) + (p0.z + p0.w)) + ((p1.x + p1.y) + (p1.z + p1.w)) +
                 ((p2.x + p2.y) + (p2.z + p2.w)) + ((p3.x + p3.y) + (p3.z + p3.w));
      }
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 9);
#pragma unroll 1
    for (int r = r0; r < r1; r += SDPI) {
      const int nr = min(SDPI, r1 - r);
      const uint8_t* st = acquire();
      if (!ctl->abort) {
#pragma unroll 1
        for (int rr = cw; rr < nr; rr += NCW) {
          const uint8_t* row = st + (size_t)rr * L.SDR;
#pragma unroll 1
          for (int tc = 0; tc < T; tc += TK) {
            const int nt = min(TK, T - tc);
            float rs[TK];
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) rs[tt] = 0.f;
#pragma unroll 1
            for (int cc = lane; cc < Is / 16; cc += 32) {
              const uint4 cw4 = *reinterpret_cast<const uint4*>(row + cc * 16);
              const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + Is + (cc >> 2) * 4));
              float2 q[8];
              unpack_int8_word(cw4.x, q[0], q[1]);
              unpack_int8_word(cw4.y, q[2], q[3]);
              unpack_int8_word(cw4.z, q[4], q[5]);
              unpack_int8_word(cw4.w, q[6], q[7]);
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                if (tt < nt) {
                  const float4* hv = reinterpret_cast<const float4*>(hsn + (size_t)(tc + tt) * Is + cc * 16);
                  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                  for (int m = 0; m < 4; ++m) {
                    const float4 h4 = hv[m];
                    acc = __ffma2_rn(q[2 * m], make_float2(h4.x, h4.y), acc);
                    acc = __ffma2_rn(q[2 * m + 1], make_float2(h4.z, h4.w), acc);
                  }
                  rs[tt] += sb.x * (acc.x + acc.y) + sb.y * hss[(tc + tt) * (Is / 16) + cc];
                }
              }
            }
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) rs[tt] = warp_sum(rs[tt]);
            if (lane == 0)
#pragma unroll 1
              for (int tt = 0; tt < nt; ++tt) shs[(tc + tt) * (r1 - r0) + (r + rr - r0)] = rs[tt];
          }
        }
      }
      release();
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 10);

    // ---- B: routed segments
    const int nseg = ctl->nseg;
#pragma unroll 1
    for (int sgi = 0; sgi < nseg; ++sgi) {
      const int u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi], ne = ctl->seg_n[sgi];
      const int units = u1 - u0;
      const uint8_t* toks = ctl->seg_tok[sgi];
      // gate/up -> h, a pair of units per warp
      if (sgi == 0) wstamp(a, cw, 0);
#pragma unroll 1
      for (int u = u0; u < u1; u += UPI) {
        const int nu = min(UPI, u1 - u);
        const uint8_t* st = acquire();
        if (!ctl->abort) {
          // pairs are numbered across the whole segment so that consecutive items go to different warps
          const int pbase = (u - u0) >> 1;
#pragma unroll 1
          for (int pr = (cw - pbase % NCW + NCW) % NCW; pr * 2 < nu; pr += NCW) {
            if (sgi == 0) wstamp(a, cw, 1);
            const uint8_t* ub = st + (size_t)(2 * pr) * L.EU;
            const int nvalid = (2 * pr + 1 < nu) ? 4 : 2;
            const int ul = u + 2 * pr - u0;
#pragma unroll 1
            for (int tc = 0; tc < ne; tc += TK) {
              const int nt = min(TK, ne - tc);
              const DotR<4, TK> d = dot_rows<H, 4, TK, false>(ub, ub + H / 2, ub + L.EU, ub + L.EU + H / 2,
                                                              ub + H, ub + H + L.GB * 4, ub + L.EU + H,
                                                              ub + L.EU + H + L.GB * 4, nvalid, xh, xs, toks[tc],
                                                              toks[tc + nt - 1], nt);
              if (lane < 2 * TK) {
                const int tt = lane >> 1, k = lane & 1;
                float g = 0.f, up = 0.f;
#pragma unroll
                for (int q = 0; q < TK; ++q)
                  if (q == tt) { g = k ? d.v[q][2] : d.v[q][0]; up = k ? d.v[q][3] : d.v[q][1]; }
                if (tt < nt && 2 * k < nvalid) hseg[(tc + tt) * units + ul + k] = silu_fast(g) * up;
              }
            }
            if (sgi == 0) wstamp(a, cw, 2);
          }
        }
        release();
      }
      named_bar(BAR_C, CT);
      if (ctid == 0 && sgi == 0) stamp(a, 7);
      if (sgi == 0) wstamp(a, cw, 3);
      // down: per group, the (s,b) block then the unit columns; each thread owns 4 output rows
      const int hq = ctid;
      const bool has_q = hq < H / 4;
      const bool in_regs = ne <= TK;   // all tokens' partial sums stay in registers across the segment
      float4 pacc[TK];
#pragma unroll
      for (int tt = 0; tt < TK; ++tt) pacc[tt] = make_float4(0.f, 0.f, 0.f, 0.f);
      bool first = true;
      const size_t slot0 = ((size_t)cta * DEC_MAXSEG + sgi) * T;
#pragma unroll 1
      for (int g = u0 / 64; g * 64 < u1; ++g) {
        float2 sbq[4];
        {
          const uint8_t* st = acquire();
          if (!ctl->abort && has_q) {
            const uint4 raw = *reinterpret_cast<const uint4*>(st + (size_t)hq * 16);
            sbq[0] = h2f(raw.x); sbq[1] = h2f(raw.y); sbq[2] = h2f(raw.z); sbq[3] = h2f(raw.w);
          }
          release();
        }
        const int ga = max(u0, g * 64), gb = min(u1, g * 64 + 64);
#pragma unroll 1
        for (int u = ga; u < gb; u += DPI) {
          const int nu = min(DPI, gb - u);
          const uint8_t* st = acquire();
          if (!ctl->abort && has_q) {
#pragma unroll 1
            for (int tc = 0; tc < ne; tc += TK) {
              const int nt = min(TK, ne - tc);
              float2 acc[TK][2];
              float hsum[TK];
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                acc[tt][0] = acc[tt][1] = make_float2(0.f, 0.f);
                hsum[tt] = 0.f;
              }
              const float* hrow = hseg + (size_t)tc * units + (u - u0);
#pragma unroll 4
              for (int k = 0; k < nu; ++k) {
                const uint32_t hw = *reinterpret_cast<const uint16_t*>(st + (size_t)k * L.DCB + hq * 2);
                float2 q01, q23;
                unpack_int4_quad(hw, q01, q23);
#pragma unroll
                for (int tt = 0; tt < TK; ++tt) {
                  if (tt < nt) {
                    const float h = hrow[tt * units + k];
                    acc[tt][0] = __ffma2_rn(q01, make_float2(h, h), acc[tt][0]);
                    acc[tt][1] = __ffma2_rn(q23, make_float2(h, h), acc[tt][1]);
                    hsum[tt] += h;
                  }
                }
              }
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                if (tt < nt) {
                  const float w = ctl->seg_w[sgi][tc + tt];
                  float4 v;
                  v.x = w * (sbq[0].x * acc[tt][0].x + sbq[0].y * hsum[tt]);
                  v.y = w * (sbq[1].x * acc[tt][0].y + sbq[1].y * hsum[tt]);
                  v.z = w * (sbq[2].x * acc[tt][1].x + sbq[2].y * hsum[tt]);
                  v.w = w * (sbq[3].x * acc[tt][1].y + sbq[3].y * hsum[tt]);
                  if (in_regs) {
                    pacc[tt].x += v.x; pacc[tt].y += v.y; pacc[tt].z += v.z; pacc[tt].w += v.w;
                  } else {
                    float4* dst = reinterpret_cast<float4*>(a.partial + (slot0 + tc + tt) * H + 4 * hq);
                    if (!first) {
                      const float4 o = __ldcg(dst);
                      v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
                    }
                    __stcg(dst, v);
                  }
                }
              }
            }
          }
          first = false;
          release();
        }
      }
      if (in_regs && !ctl->abort && has_q) {
#pragma unroll
        for (int tt = 0; tt < TK; ++tt)
          if (tt < ne) __stcg(reinterpret_cast<float4*>(a.partial + (slot0 + tt) * H + 4 * hq), pacc[tt]);
      }
      named_bar(BAR_C, CT);
    }
    if (ctid == 0) stamp(a, 8);

    // ---- D: all partials finished -> fixed-order reduction of this CTA's rows
    if (ctid == 0) {
      __threadfence();
      atomicAdd(&a.counters[2], 1u);
      if (!ctl->abort && !spin_geq(&a.counters[2], (uint32_t)G, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_PARTIAL);
      stamp(a, 11);
    }
    // while thread 0 waits for every CTA: per token, the list of partial-sum slots that hold it
#pragma unroll 1
      for (int t = cw - 1; cw > 0 && t < T; t += NCW - 1) {
        int n = 0;
#pragma unroll 1
        for (int c0 = 0; c0 < G; c0 += 32) {
          const int c = c0 + lane;
          uint32_t cnt = 0, sl[2] = {0u, 0u};
          if (c < G) {
            const int a0 = ctl->tab_a0[c], ns = min((int)ctl->tab_n[c], 2);
#pragma unroll
            for (int sg = 0; sg < 2; ++sg) {
              if (sg < ns) {
                const uint32_t msk = ctl->act_mask[a0 + sg];
                if ((msk >> t) & 1u) {
                  sl[cnt] = ((uint32_t)c * DEC_MAXSEG + sg) * T + __popc(msk & ((1u << t) - 1u));
                  ++cnt;
                }
              }
            }
          }
          uint32_t incl = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += v;
          }
          const int pos = n + (int)(incl - cnt);
          if (cnt > 0) ctl->slot[t][pos] = (uint16_t)sl[0];
          if (cnt > 1) ctl->slot[t][pos + 1] = (uint16_t)sl[1];
          n += (int)__shfl_sync(FULL, incl, 31);
        }
        if (lane == 0) ctl->nslot[t] = n;
      }
    named_bar(BAR_C, CT);
    if (!ctl->abort) {
      const int nr = r1 - r0;
#pragma unroll 1
      for (int pi = cw; pi < T * nr; pi += NCW) {
        const int t = pi / nr, rr = pi % nr, row = r0 + rr;
        // every partial this lane needs is loaded before any is added (independent L2 reads in flight)
        const int ns = ctl->nslot[t];
        float v[2 * DEC_MAXGRID / 32];
#pragma unroll
        for (int k = 0; k < 2 * DEC_MAXGRID / 32; ++k) {
          const int q = lane + 32 * k;
          v[k] = q < ns ? __ldcg(a.partial + (size_t)ctl->slot[t][q] * H + row) : 0.f;
        }
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 2 * DEC_MAXGRID / 32; ++k) acc += v[k];
        // rare: a CTA whose unit range touches more than two experts
#pragma unroll 1
        for (int c = lane; c < G; c += 32) {
          const int a0 = ctl->tab_a0[c], ns = ctl->tab_n[c];
#pragma unroll 1
          for (int sg = 2; sg < ns; ++sg) {
            const uint32_t msk = ctl->act_mask[a0 + sg];
            if ((msk >> t) & 1u) {
              const int tl = __popc(msk & ((1u << t) - 1u));
              acc += __ldcg(a.partial + (((size_t)c * DEC_MAXSEG + sg) * T + tl) * H + row);
            }
          }
        }
        acc = warp_sum(acc);
        if (lane == 0) {
          float v = acc + ctl->sg[t] * shs[t * nr + rr];
          if (a.gamma) v += __half2float(__ushort_as_half(a.x[(size_t)t * H + row]));
          a.out[(size_t)t * H + row] = __half_as_ushort(__float2half_rn(v));
        }
      }
    }
    named_bar(BAR_C, CT);
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    stamp(a, 12);
    __threadfence();
    const uint32_t prev = atomicAdd(&a.counters[3], 1u);
    if (prev == (uint32_t)G - 1) {
      a.counters[0] = 0; a.counters[1] = 0; a.counters[2] = 0;
      __threadfence();
      a.counters[3] = 0;
    }
  }
}

template <int H>
int hseg_bound(const MoeLayout& L, int T, int grid) {
  int best = 0;
  const int TK = T * L.K;
#pragma unroll 1
  for (int n = 1; n <= T; ++n) {
    long long U = (long long)TK - n + 1;
    if (U > L.E) U = L.E;
    long long units = (U * L.I + grid - 1) / grid + 1;
    if (units > L.I) units = L.I;
    long long v = units * n;
    if (v > best) best = (int)v;
  }
  return best;
}

}  // namespace

size_t decode_partial_floats(const MoeLayout& L, int grid, int T) {
  return (size_t)grid * DEC_MAXSEG * T * L.H;
}

bool decode_plan(const MoeLayout& L, int T, int grid, int max_smem, DecodeLaunch* out) {
  if (grid > DEC_MAXGRID) return false;
  DecodeLaunch pl;
  pl.grid = grid;
  pl.hseg_floats = hseg_bound<0>(L, T, grid);
  const Smem m = smem_map(L, T, grid, pl.hseg_floats);
  const int upi = T <= 4 ? 8 : 4;
  int SS = (int)(upi * L.EU);
  if (SS < 4 * L.H) SS = 4 * L.H;
  if ((int)(2 * L.SU) > SS) SS = (int)(2 * L.SU);
  if ((int)L.RR > SS) SS = (int)L.RR;
  if ((int)L.SDR > SS) SS = (int)L.SDR;
  SS = (SS + 127) & ~127;
  int NS = (max_smem - m.ring) / SS;
  if (NS > DEC_MAXNS) NS = DEC_MAXNS;
  if (NS < 3) return false;
  pl.NS = NS;
  pl.SS = SS;
  pl.smem = m.ring + NS * SS;
  *out = pl;
  return true;
}

template <class SH, int TK>
static cudaError_t launch_s(const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  auto kern = k_decode<SH, TK>;
  // raise the dynamic shared-memory limit once per process and instantiation (a per-function setting)
  static int configured = 0;
  if (configured < pl.smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    configured = pl.smem > 232448 ? pl.smem : 232448;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(DEC_THREADS);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, pl.NS, pl.SS, pl.hseg_floats);
}

template <class SH>
static bool is_shape(const MoeLayout& L) {
  return L.H == SH::H && L.E == SH::E && L.K == SH::K && L.I == SH::I && L.Is == SH::Is;
}

bool decode_supported(const MoeLayout& L) { return is_shape<ShapeProd>(L) || is_shape<ShapeTiny>(L); }

cudaError_t decode_launch(const MoeLayout& L, const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  const bool small = a.T == 1;
  if (is_shape<ShapeProd>(L)) return small ? launch_s<ShapeProd, 1>(a, pl, st) : launch_s<ShapeProd, 2>(a, pl, st);
  if (is_shape<ShapeTiny>(L)) return small ? launch_s<ShapeTiny, 1>(a, pl, st) : launch_s<ShapeTiny, 2>(a, pl, st);
  return cudaErrorNotSupported;
}

}  // namespace moe
