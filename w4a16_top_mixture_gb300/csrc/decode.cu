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
constexpr int BAR_C = 1;       // named barrier of the consumer warps
constexpr uint32_t FULL = 0xFFFFFFFFu;

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
  uint32_t emask[512];
  uint16_t act_e[512];
  uint32_t act_mask[512];
  int warp_tot[NCW];
};
constexpr int CTL_BYTES = (sizeof(Ctl) + 127) & ~127;

struct Smem {   // byte offsets of the dynamic shared-memory regions
  int xp, xs, hss, hseg, shs, ring;
};

__host__ __device__ inline Smem smem_map(const MoeLayout& L, int T, int grid, int hseg_floats) {
  Smem m;
  int o = CTL_BYTES;
  m.xp = o;
  int xbytes = T * L.H * 4, hsbytes = T * L.Is * 4;
  o += ((xbytes > hsbytes ? xbytes : hsbytes) + 127) & ~127;
  m.xs = o;   o += (T * L.NCH * 4 + 127) & ~127;
  m.hss = o;  o += (T * (L.Is / 16) * 4 + 127) & ~127;
  m.hseg = o; o += (hseg_floats * 4 + 127) & ~127;
  int rpc = (L.H + grid - 1) / grid;
  m.shs = o;  o += (T * rpc * 4 + 127) & ~127;
  m.ring = o;
  return m;
}

__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)(((long long)n * c) / G); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void set_error(const DecodeArgs& a, Ctl* ctl, uint32_t bit) {
  atomicOr(a.status, bit);
  ctl->abort = 1;
}

// Dot products of NR rows (a warp's work item) with TK tokens at a time. Codes: int4 rows in canonical
// packing (INT8 = false) or permuted int8 rows. Lane l covers the 32-column chunks c = l + LW*p. emit(tc,
// nt, rs) is called with the warp-reduced row sums rs[tt][r] = sum_c (s_g(c) * dot_c + b_g(c) * xsum_c).
template <int H, int NR, int TK, bool INT8, typename Emit>
__device__ __forceinline__ void rows_dot(const uint8_t* const* rowp, const uint8_t* const* sbp, int nvalid,
                                         const float4* __restrict__ xp, const float* __restrict__ xs,
                                         const uint8_t* toks, int ntok, Emit emit) {
  constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  const int lane = threadIdx.x & 31;
  for (int tc = 0; tc < ntok; tc += TK) {
    const int nt = min(TK, ntok - tc);
    int tix[TK];
#pragma unroll
    for (int tt = 0; tt < TK; ++tt) tix[tt] = tt < nt ? (toks ? (int)toks[tc + tt] : tc + tt) : 0;
    float rs[TK][NR];
#pragma unroll
    for (int tt = 0; tt < TK; ++tt)
#pragma unroll
      for (int r = 0; r < NR; ++r) rs[tt][r] = 0.f;
    if (lane < LW) {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int c = lane + LW * p;
        float2 acc[TK][NR];
#pragma unroll
        for (int tt = 0; tt < TK; ++tt)
#pragma unroll
          for (int r = 0; r < NR; ++r) acc[tt][r] = make_float2(0.f, 0.f);
        uint4 c4[NR];   // int4: the chunk's 16 bytes (32 codes) of each row
        if (!INT8) {
#pragma unroll
          for (int r = 0; r < NR; ++r)
            c4[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rowp[r] + c * 16)
                               : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // int8: one 16-byte load (16 codes) per half chunk
          uint4 cw[NR];
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (INT8)
              cw[r] = r < nvalid ? *reinterpret_cast<const uint4*>(rowp[r] + ((p * 2 + hh) * LW + lane) * 16)
                                 : make_uint4(0x80808080u, 0x80808080u, 0x80808080u, 0x80808080u);
            else
              cw[r] = c4[r];
          }
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = hh * 2 + jj;   // 8-column block within the chunk
            float4 xa[TK], xb[TK];
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) {
              if (tt < nt) {
                const int base = ((tix[tt] * P + p) * 8 + j * 2) * LW + lane;
                xa[tt] = xp[base];
                xb[tt] = xp[base + LW];
              } else {
                xa[tt] = make_float4(0.f, 0.f, 0.f, 0.f);
                xb[tt] = xa[tt];
              }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
              float2 q[4];
              if (INT8) {
                const uint32_t w0 = jj == 0 ? cw[r].x : cw[r].z;
                const uint32_t w1 = jj == 0 ? cw[r].y : cw[r].w;
                unpack_int8_pair(w0, w1, q);
              } else {
                const uint32_t w = j == 0 ? cw[r].x : j == 1 ? cw[r].y : j == 2 ? cw[r].z : cw[r].w;
                unpack_int4_word(w, q);
              }
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                acc[tt][r] = __ffma2_rn(q[0], make_float2(xa[tt].x, xa[tt].y), acc[tt][r]);
                acc[tt][r] = __ffma2_rn(q[1], make_float2(xa[tt].z, xa[tt].w), acc[tt][r]);
                acc[tt][r] = __ffma2_rn(q[2], make_float2(xb[tt].x, xb[tt].y), acc[tt][r]);
                acc[tt][r] = __ffma2_rn(q[3], make_float2(xb[tt].z, xb[tt].w), acc[tt][r]);
              }
            }
          }
        }
        // per-chunk affine: s * sum(q x) + b * sum(x)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r < nvalid) {
            const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(sbp[r] + (c >> 1) * 4));
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) {
              const float X = xs[(tix[tt] * P + p) * LW + lane];
              rs[tt][r] += sb.x * (acc[tt][r].x + acc[tt][r].y) + sb.y * X;
            }
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TK; ++tt)
#pragma unroll
      for (int r = 0; r < NR; ++r) rs[tt][r] = warp_sum(rs[tt][r]);
    emit(tc, nt, rs);
  }
}

template <int H, int TK>
__global__ void __launch_bounds__(DEC_THREADS, 1) k_decode(MoeLayout L, DecodeArgs a, int NS, int SS,
                                                           int hseg_floats) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCH = H / 32, LW = NCH < 32 ? NCH : 32, P = (NCH + 31) / 32;
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = a.T, E = L.E, K = L.K, I = L.I, Is = L.Is;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  const Smem sm = smem_map(L, T, G, hseg_floats);
  float4* xp = reinterpret_cast<float4*>(smem + sm.xp);
  float* xs = reinterpret_cast<float*>(smem + sm.xs);
  float* hsp = reinterpret_cast<float*>(smem + sm.xp);   // shared-expert h (aliases x after phase B)
  float* hss = reinterpret_cast<float*>(smem + sm.hss);
  float* hseg = reinterpret_cast<float*>(smem + sm.hseg);
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

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int n = 0;
      const uint64_t pol = policy_evict_first();
      auto issue = [&](const uint8_t* src, uint32_t bytes) -> bool {
        if (ctl->abort) return false;
        const int s = n % NS;
        if (n >= NS && !mbar_wait(&ctl->empty[s], ((n / NS) - 1) & 1, a.timeout_ns)) {
          set_error(a, ctl, ERR_WAIT_EMPTY);
          return false;
        }
        mbar_expect_tx(&ctl->full[s], bytes);
        bulk_g2s_hint(ring + (size_t)s * SS, src, bytes, &ctl->full[s], pol);
        ++n;
        return true;
      };
      bool ok = true;
      for (int r = ra; ok && r < rb; r += RPI) {
        const int nr = min(RPI, rb - r);
        ok = issue(a.router + (size_t)r * L.RR, (uint32_t)(nr * L.RR));
      }
      for (int u = sa; ok && u < sbn; u += SPI) {
        const int nu = min(SPI, sbn - u);
        ok = issue(a.sh_gu + (size_t)u * L.SU, (uint32_t)(nu * L.SU));
      }
      if (ok && !mbar_wait(&ctl->route_ready, 0, a.timeout_ns * 4)) {
        set_error(a, ctl, ERR_WAIT_ROUTE);
        ok = false;
      }
      if (ok && ctl->abort) ok = false;
      const int nseg = ok ? ctl->nseg : 0;
      for (int sgi = 0; ok && sgi < nseg; ++sgi) {
        const int e = ctl->seg_e[sgi], u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi];
        const uint8_t* gu = a.ex_gu + (size_t)e * L.exgu_expert;
        for (int u = u0; ok && u < u1; u += UPI)
          ok = issue(gu + (size_t)u * L.EU, (uint32_t)(min(UPI, u1 - u) * L.EU));
        const uint8_t* dn = a.ex_dn + (size_t)e * L.exdn_expert;
        for (int g = u0 / 64; ok && g * 64 < u1; ++g) {
          const uint8_t* blk = dn + (size_t)g * L.DB;
          ok = issue(blk, (uint32_t)L.DSB);
          const int ga = max(u0, g * 64), gb = min(u1, g * 64 + 64);
          for (int u = ga; ok && u < gb; u += DPI)
            ok = issue(blk + L.DSB + (size_t)(u - g * 64) * L.DCB, (uint32_t)(min(DPI, gb - u) * L.DCB));
        }
      }
      for (int r = r0; ok && r < r1; r += SDPI)
        ok = issue(a.sh_dn + (size_t)r * L.SDR, (uint32_t)(min(SDPI, r1 - r) * L.SDR));
      // drain: every issued copy must have landed before the CTA may leave
      for (int m = max(0, n - NS); m < n; ++m)
        if (!mbar_wait(&ctl->full[m % NS], (m / NS) & 1, a.timeout_ns)) atomicOr(a.status, ERR_WAIT_FULL);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    int it = 0;   // item counter, mirrors the producer's
    auto acquire = [&]() -> const uint8_t* {
      const int s = it % NS;
      if (!ctl->abort && !mbar_wait(&ctl->full[s], (it / NS) & 1, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_FULL);
      return ring + (size_t)s * SS;
    };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[it % NS]);
      ++it;
    };

    // ---- x prologue: (RMSNorm) -> fp16 -> fp32, permuted for the row dots, plus 32-column sums
    for (int t = cw; t < T; t += NCW) {
      const uint16_t* xr = a.x + (size_t)t * H;
      float v[P][32];
      float ss = 0.f;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int c = lane + LW * p;
        if (lane < LW) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 raw = *reinterpret_cast<const uint4*>(xr + c * 32 + q4 * 8);
            const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float2 f = __half22float2(hv[k]);
              v[p][q4 * 8 + 2 * k] = f.x;
              v[p][q4 * 8 + 2 * k + 1] = f.y;
            }
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) ss += v[p][k] * v[p][k];
        }
      }
      if (a.gamma) {
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / (float)H + a.eps);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const int c = lane + LW * p;
          if (lane < LW) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const float g = __half2float(__ushort_as_half(a.gamma[c * 32 + k]));
              v[p][k] = __half2float(__float2half_rn(v[p][k] * rn * g));
            }
          }
        }
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if (lane < LW) {
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k) sum += v[p][k];
          xs[(t * P + p) * LW + lane] = sum;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float* b8 = &v[p][8 * j];
            const int base = ((t * P + p) * 8 + j * 2) * LW + lane;
            xp[base] = make_float4(b8[0], b8[4], b8[1], b8[5]);
            xp[base + LW] = make_float4(b8[2], b8[6], b8[3], b8[7]);
          }
        }
      }
    }
    named_bar(BAR_C, CT);

    // ---- A1: router rows
    for (int r = ra; r < rb; r += RPI) {
      const int nr = min(RPI, rb - r);
      const uint8_t* st = acquire();
      if (!ctl->abort) {
        for (int rr = cw; rr < nr; rr += NCW) {
          const uint8_t* rowp[1] = {st + (size_t)rr * L.RR};
          const uint8_t* sbp[1] = {st + (size_t)rr * L.RR + H};
          const int row = r + rr;
          rows_dot<H, 1, TK, true>(rowp, sbp, 1, xp, xs, nullptr, T, [&](int tc, int nt, float (*rs)[1]) {
            if (lane == 0)
              for (int tt = 0; tt < nt; ++tt) a.logits[(size_t)(tc + tt) * (E + 1) + row] = rs[tt][0];
          });
        }
      }
      release();
    }
    named_bar(BAR_C, CT);
    if (ctid == 0 && !(a.skip_arrive && cta == 0)) {
      __threadfence();
      atomicAdd(&a.counters[0], 1u);
    }

    // ---- R: routing (every CTA, every token)
    if (ctid == 0 && !ctl->abort && !spin_geq(&a.counters[0], (uint32_t)G, a.timeout_ns))
      set_error(a, ctl, ERR_WAIT_LOGITS);
    named_bar(BAR_C, CT);
    __threadfence();
    if (!ctl->abort) {
      const int EPL = (E + 31) / 32;
      for (int t = cw; t < T; t += NCW) {
        const float* lg = a.logits + (size_t)t * (E + 1);
        uint32_t key[16];
        float val[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = lane * EPL + i;
          const bool in = i < EPL && e < E;
          const float v = in ? __ldcg(lg + e) : 0.f;
          const uint32_t b = __float_as_uint(v);
          key[i] = in ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
          val[i] = v;
        }
        int my_idx = -1;
        float my_logit = 0.f;
        for (int j = 0; j < K; ++j) {
          uint32_t best = 0;
          int bi = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (key[i] > best) { best = key[i]; bi = i; }
          const uint32_t m = __reduce_max_sync(FULL, best);
          const int win = __ffs(__ballot_sync(FULL, best == m)) - 1;
          float lv = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i == bi) lv = val[i];
          if (lane == win) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i == bi) key[i] = 0u;
          }
          const int sel = __shfl_sync(FULL, lane * EPL + bi, win);
          const float sl = __shfl_sync(FULL, lv, win);
          if (lane == j) { my_idx = sel; my_logit = sl; }
        }
        const float mx = __shfl_sync(FULL, my_logit, 0);
        const float ex = lane < K ? expf(my_logit - mx) : 0.f;
        const float Z = warp_sum(ex);
        int rank = 0;
        for (int i = 0; i < K; ++i) {
          const int oi = __shfl_sync(FULL, my_idx, i);
          rank += (lane < K && oi < my_idx) ? 1 : 0;
        }
        if (lane < K) {
          ctl->ids[t][rank] = my_idx;
          ctl->wts[t][rank] = ex / Z;
        }
        if (lane == 0) {
          const float g = __ldcg(lg + E);
          ctl->sg[t] = 1.0f / (1.0f + expf(-g));
        }
      }
    }
    named_bar(BAR_C, CT);
    // bucketing: token masks per expert, active experts in ascending order
    for (int e = ctid; e < E; e += CT) ctl->emask[e] = 0u;
    named_bar(BAR_C, CT);
    if (!ctl->abort)
      for (int p = ctid; p < T * K; p += CT) atomicOr(&ctl->emask[ctl->ids[p / K][p % K]], 1u << (p / K));
    named_bar(BAR_C, CT);
    {
      const uint32_t msk = ctid < E ? ctl->emask[ctid] : 0u;
      const uint32_t bal = __ballot_sync(FULL, msk != 0u);
      if (lane == 0) ctl->warp_tot[cw] = __popc(bal);
      named_bar(BAR_C, CT);
      int base = 0;
      for (int w = 0; w < cw; ++w) base += ctl->warp_tot[w];
      if (msk != 0u) {
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        ctl->act_e[pos] = (uint16_t)ctid;
        ctl->act_mask[pos] = msk;
      }
      if (ctid == CT - 1) ctl->U = base + __popc(bal);
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) {
      const int U = ctl->U;
      const int N = U * I;
      const int lo = range_lo(N, cta, G), hi = range_lo(N, cta + 1, G);
      int nseg = 0;
      for (int aa = lo / I; aa * I < hi && lo < hi; ++aa) {
        if (nseg == DEC_MAXSEG) { set_error(a, ctl, ERR_SEGMENTS); break; }
        const int e = ctl->act_e[aa];
        const uint32_t msk = ctl->act_mask[aa];
        ctl->seg_a[nseg] = aa;
        ctl->seg_e[nseg] = e;
        ctl->seg_u0[nseg] = max(lo, aa * I) - aa * I;
        ctl->seg_u1[nseg] = min(hi, (aa + 1) * I) - aa * I;
        int n = 0;
        for (int t = 0; t < T; ++t) {
          if (msk & (1u << t)) {
            ctl->seg_tok[nseg][n] = (uint8_t)t;
            float wv = 0.f;
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
      if (cta == 0 && a.rec_ids) {
        for (int t = 0; t < T; ++t) {
          for (int j = 0; j < K; ++j) {
            a.rec_ids[t * K + j] = ctl->ids[t][j];
            a.rec_w[t * K + j] = ctl->wts[t][j];
          }
          a.rec_sg[t] = ctl->sg[t];
        }
      }
      mbar_arrive(&ctl->route_ready);
    }
    named_bar(BAR_C, CT);

    // ---- A2: shared-expert gate/up units (pairs of units per warp)
    for (int u = sa; u < sbn; u += SPI) {
      const int nu = min(SPI, sbn - u);
      const uint8_t* st = acquire();
      if (!ctl->abort) {
        for (int pr = cw; pr * 2 < nu; pr += NCW) {
          const uint8_t* ub = st + (size_t)(2 * pr) * L.SU;
          const uint8_t* rowp[4] = {ub, ub + H, ub + L.SU, ub + L.SU + H};
          const uint8_t* sbp[4] = {ub + 2 * H, ub + 2 * H + L.GB * 4, ub + L.SU + 2 * H,
                                   ub + L.SU + 2 * H + L.GB * 4};
          const int nvalid = (2 * pr + 1 < nu) ? 4 : 2;
          const int i0 = u + 2 * pr;
          rows_dot<H, 4, TK, true>(rowp, sbp, nvalid, xp, xs, nullptr, T, [&](int tc, int nt, float (*rs)[4]) {
            if (lane == 0)
              for (int tt = 0; tt < nt; ++tt) {
                a.hs[(size_t)(tc + tt) * Is + i0] = silu_f(rs[tt][0]) * rs[tt][1];
                if (nvalid == 4) a.hs[(size_t)(tc + tt) * Is + i0 + 1] = silu_f(rs[tt][2]) * rs[tt][3];
              }
          });
        }
      }
      release();
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) {
      __threadfence();
      atomicAdd(&a.counters[1], 1u);
    }

    // ---- B: routed segments
    const int nseg = ctl->nseg;
    for (int sgi = 0; sgi < nseg; ++sgi) {
      const int u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi], ne = ctl->seg_n[sgi];
      const int units = u1 - u0;
      const uint8_t* toks = ctl->seg_tok[sgi];
      // gate/up -> h
      for (int u = u0; u < u1; u += UPI) {
        const int nu = min(UPI, u1 - u);
        const uint8_t* st = acquire();
        if (!ctl->abort) {
          for (int pr = cw; pr * 2 < nu; pr += NCW) {
            const uint8_t* ub = st + (size_t)(2 * pr) * L.EU;
            const uint8_t* rowp[4] = {ub, ub + H / 2, ub + L.EU, ub + L.EU + H / 2};
            const uint8_t* sbp[4] = {ub + H, ub + H + L.GB * 4, ub + L.EU + H, ub + L.EU + H + L.GB * 4};
            const int nvalid = (2 * pr + 1 < nu) ? 4 : 2;
            const int ul = u + 2 * pr - u0;
            rows_dot<H, 4, TK, false>(rowp, sbp, nvalid, xp, xs, toks, ne, [&](int tc, int nt, float (*rs)[4]) {
              if (lane == 0)
                for (int tt = 0; tt < nt; ++tt) {
                  hseg[(tc + tt) * units + ul] = silu_f(rs[tt][0]) * rs[tt][1];
                  if (nvalid == 4) hseg[(tc + tt) * units + ul + 1] = silu_f(rs[tt][2]) * rs[tt][3];
                }
            });
          }
        }
        release();
      }
      named_bar(BAR_C, CT);
      // down: per group, the (s,b) block then the unit columns
      const int hq = ctid;   // row quad
      const bool has_q = hq < H / 4;
      bool first = true;
      const size_t slot0 = ((size_t)cta * DEC_MAXSEG + sgi) * T;
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
        for (int u = ga; u < gb; u += DPI) {
          const int nu = min(DPI, gb - u);
          const uint8_t* st = acquire();
          if (!ctl->abort && has_q) {
            for (int tc = 0; tc < ne; tc += TK) {
              const int nt = min(TK, ne - tc);
              float2 acc[TK][2];
              float hsum[TK];
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                acc[tt][0] = acc[tt][1] = make_float2(0.f, 0.f);
                hsum[tt] = 0.f;
              }
              for (int k = 0; k < nu; ++k) {
                const uint32_t hw = *reinterpret_cast<const uint16_t*>(st + (size_t)k * L.DCB + hq * 2);
                float2 q01, q23;
                unpack_int4_quad(hw, q01, q23);
                const int ul = u + k - u0;
#pragma unroll
                for (int tt = 0; tt < TK; ++tt) {
                  if (tt < nt) {
                    const float h = hseg[(tc + tt) * units + ul];
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
          first = false;
          release();
        }
      }
      named_bar(BAR_C, CT);
    }

    // ---- C: shared down rows (needs every CTA's hs)
    if (ctid == 0 && !ctl->abort && !spin_geq(&a.counters[1], (uint32_t)G, a.timeout_ns))
      set_error(a, ctl, ERR_WAIT_HS);
    named_bar(BAR_C, CT);
    __threadfence();
    if (!ctl->abort) {
      // stage hs permuted in 8-blocks (0,4,1,5,2,6,3,7) and its 16-column sums
      for (int i = ctid; i < T * Is / 8; i += CT) {
        const int t = i / (Is / 8), blk = i % (Is / 8);
        const float4 lo = __ldcg(reinterpret_cast<const float4*>(a.hs + (size_t)t * Is + blk * 8));
        const float4 hi = __ldcg(reinterpret_cast<const float4*>(a.hs + (size_t)t * Is + blk * 8 + 4));
        float4* d = reinterpret_cast<float4*>(hsp + (size_t)t * Is + blk * 8);
        d[0] = make_float4(lo.x, hi.x, lo.y, hi.y);
        d[1] = make_float4(lo.z, hi.z, lo.w, hi.w);
      }
      for (int i = ctid; i < T * (Is / 16); i += CT) {
        const int t = i / (Is / 16), c = i % (Is / 16);
        const float* src = a.hs + (size_t)t * Is + c * 16;
        float s = 0.f;
        for (int k = 0; k < 16; ++k) s += __ldcg(src + k);
        hss[i] = s;
      }
    }
    named_bar(BAR_C, CT);
    for (int r = r0; r < r1; r += SDPI) {
      const int nr = min(SDPI, r1 - r);
      const uint8_t* st = acquire();
      if (!ctl->abort) {
        for (int rr = cw; rr < nr; rr += NCW) {
          const uint8_t* row = st + (size_t)rr * L.SDR;
          for (int tc = 0; tc < T; tc += TK) {
            const int nt = min(TK, T - tc);
            float rs[TK];
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) rs[tt] = 0.f;
            for (int cc = lane; cc < Is / 16; cc += 32) {
              const uint4 cw4 = *reinterpret_cast<const uint4*>(row + cc * 16);
              const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + Is + (cc >> 2) * 4));
              float2 q0[4], q1[4];
              unpack_int8_pair(cw4.x, cw4.y, q0);
              unpack_int8_pair(cw4.z, cw4.w, q1);
#pragma unroll
              for (int tt = 0; tt < TK; ++tt) {
                if (tt < nt) {
                  const float4* hv = reinterpret_cast<const float4*>(hsp + (size_t)(tc + tt) * Is + cc * 16);
                  const float4 A = hv[0], B = hv[1], C = hv[2], D = hv[3];
                  float2 acc = make_float2(0.f, 0.f);
                  acc = __ffma2_rn(q0[0], make_float2(A.x, A.y), acc);
                  acc = __ffma2_rn(q0[1], make_float2(A.z, A.w), acc);
                  acc = __ffma2_rn(q0[2], make_float2(B.x, B.y), acc);
                  acc = __ffma2_rn(q0[3], make_float2(B.z, B.w), acc);
                  acc = __ffma2_rn(q1[0], make_float2(C.x, C.y), acc);
                  acc = __ffma2_rn(q1[1], make_float2(C.z, C.w), acc);
                  acc = __ffma2_rn(q1[2], make_float2(D.x, D.y), acc);
                  acc = __ffma2_rn(q1[3], make_float2(D.z, D.w), acc);
                  rs[tt] += sb.x * (acc.x + acc.y) + sb.y * hss[(tc + tt) * (Is / 16) + cc];
                }
              }
            }
#pragma unroll
            for (int tt = 0; tt < TK; ++tt) rs[tt] = warp_sum(rs[tt]);
            if (lane == 0)
              for (int tt = 0; tt < nt; ++tt) shs[(tc + tt) * (r1 - r0) + (r + rr - r0)] = rs[tt];
          }
        }
      }
      release();
    }
    named_bar(BAR_C, CT);

    // ---- D: all partials finished -> fixed-order reduction of this CTA's rows
    if (ctid == 0) {
      __threadfence();
      atomicAdd(&a.counters[2], 1u);
      if (!ctl->abort && !spin_geq(&a.counters[2], (uint32_t)G, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_PARTIAL);
    }
    named_bar(BAR_C, CT);
    __threadfence();
    if (!ctl->abort) {
      const int nr = r1 - r0;
      const int U = ctl->U;
      const int N = U * I;
      for (int pi = cw; pi < T * nr; pi += NCW) {
        const int t = pi / nr, rr = pi % nr, row = r0 + rr;
        float acc = 0.f;
        for (int c = lane; c < G; c += 32) {
          const int lo = range_lo(N, c, G), hi = range_lo(N, c + 1, G);
          if (lo >= hi) continue;
          const int a0 = lo / I;
          for (int aa = a0; aa * I < hi && aa - a0 < DEC_MAXSEG; ++aa) {
            const uint32_t msk = ctl->act_mask[aa];
            if (msk & (1u << t)) {
              const int tl = __popc(msk & ((1u << t) - 1u));
              const size_t slot = ((size_t)c * DEC_MAXSEG + (aa - a0)) * T + tl;
              acc += __ldcg(a.partial + slot * H + row);
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

template <int H, int TK>
static cudaError_t launch_h(const MoeLayout& L, const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  auto kern = k_decode<H, TK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
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
  return cudaLaunchKernelEx(&cfg, kern, L, a, pl.NS, pl.SS, pl.hseg_floats);
}

cudaError_t decode_launch(const MoeLayout& L, const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  const bool small = a.T == 1;
  switch (L.H) {
    case 512: return small ? launch_h<512, 1>(L, a, pl, st) : launch_h<512, 2>(L, a, pl, st);
    case 1024: return small ? launch_h<1024, 1>(L, a, pl, st) : launch_h<1024, 2>(L, a, pl, st);
    case 2048: return small ? launch_h<2048, 1>(L, a, pl, st) : launch_h<2048, 2>(L, a, pl, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
