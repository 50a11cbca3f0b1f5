// Fused decode kernel of the W4A16 routed-MoE block (T <= 16 tokens): one persistent launch with
// one CTA per SM.
//
// Roles inside a CTA: warp 0 is the producer (one lane issues 1-D bulk copies of contiguous weight ranges
// into a ring of shared-memory stages, each guarded by a "full" and an "empty" mbarrier); warps 1..16 are
// consumers. Work a CTA owns, in stream order:
//   A1  its share of the router rows (int8)            -> logits to global, then a grid-wide arrival count
//   R   routing: every CTA waits for all logits and computes softmax -> top-k -> renormalise for every token
//       itself (identical arithmetic everywhere), buckets the (token, expert) pairs by expert and plans its
//       share of the routed units; the producer is released as soon as the plan exists
//   A2  (concurrently with R) its share of the shared-expert gate/up units -> hs to global, arrival count
//   B1  its share of all (active expert, intermediate unit) pairs: h = silu(Wg x) * (Wu x) for every token of
//       the expert, written to a global row per (expert, token) pair; arrival count
//   C   the shared expert's down projection for the CTA's own output rows (needs every CTA's hs)
//   B2  after every CTA's h is in: the routed down projection for the CTA's own output rows, every active
//       expert's rows of the down matrix against the staged h of its pairs
//   D   out = sum over the token's experts, in a fixed order, of w * y + sigmoid(g) * shared (+ residual),
//       rounded to fp16 once
// The output rows a CTA owns are its own from C to D, so no cross-CTA reduction follows the down projection.
// Every grid-wide or mbarrier wait is bounded by a timeout; a timeout records an error bit and the CTA
// drains its in-flight copies and leaves, so no wait can hang the GPU.
#include <cuda_fp16.h>
#include <mutex>
#include <stdint.h>

#include "decode.cuh"
#include "decode_dev.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int NCW = DEC_NCW;
constexpr int CT = NCW * 32;   // consumer threads
constexpr int BAR_C = 1;       // named barrier of all consumer warps
constexpr int BAR_A = 2;       // the shared-expert team
constexpr int BAR_R = 3;       // the routing team
constexpr int PMAX = DEC_TMAX * 16;   // (token, expert) pairs

struct Ctl {
  uint64_t full[DEC_MAXNS];
  uint64_t empty[DEC_MAXNS];
  uint64_t route_ready;
  volatile int abort;
  int U;                              // active experts
  int nseg;                           // segments of this CTA's routed-unit range
  int seg_a[DEC_MAXSEG], seg_u0[DEC_MAXSEG], seg_u1[DEC_MAXSEG];
  int ids[DEC_TMAX][16];
  float wts[DEC_TMAX][16];
  float sg[DEC_TMAX];
  float rn[DEC_TMAX];
  uint32_t emask[512];                // tokens routed to each expert
  uint16_t act_e[512];                // active experts, in bucket order
  uint32_t act_mask[512];
  uint16_t act_pb[513];               // first sorted pair of each active expert (act_pb[U] = number of pairs)
  uint8_t pair_tok[PMAX];             // token of each sorted pair
  float pair_w[PMAX];                 // routing weight of each sorted pair
  uint8_t tok_pair[DEC_TMAX][16];     // token t's j-th expert -> its sorted pair
  int warp_tot[NCW], warp_tot2[NCW];
  unsigned long long tclk[32];        // phase stamps (SM clock), flushed to the trace buffer at exit
  unsigned long long wclk[NCW][4];    // per-warp stamps
};
constexpr int CTL_BYTES = (sizeof(Ctl) + 127) & ~127;

struct Smem {   // byte offsets of the dynamic shared-memory regions
  int xh, xs, hst, yv, shs, ring;
};

// xh: x as int16 pairs [T][P][4 blocks][LW lanes] uint4, xs: per (token, 32-column chunk) its scale and sum
// (the activation layout of dot_rows); hst: phase C's hs [T][Is] (fp32); yv: routed down results [pair][row];
// shs: shared down results [token][row]; ring: the weight stages.
template <class LT>
__host__ __device__ inline Smem smem_map(const LT& L, int T, int grid) {
  Smem m;
  const int rows = (L.H + grid - 1) / grid;
  int o = CTL_BYTES;
  m.xh = o;   o += (T * L.H * 2 + 127) & ~127;
  m.xs = o;   o += (T * L.NCH * 8 + 127) & ~127;
  m.hst = o;  o += (T * L.Is * 4 + 127) & ~127;
  m.yv = o;   o += (T * L.K * rows * 4 + 127) & ~127;
  m.shs = o;  o += (T * rows * 4 + 127) & ~127;
  m.ring = o;
  return m;
}

// Phase stamps read the SM clock into shared memory (a few cycles, so tracing barely perturbs the kernel) and
// are written out once at exit: trace[cta*32 + slot] (slots 30 / 31: globaltimer at start / end, which place
// the CTA's clock on a common time axis) and per-warp stamps trace[grid*32 + (cta*16 + warp)*4 + k].
#define stamp(a, slot) do { if ((a).trace) ctl->tclk[(slot)] = clock64(); } while (0)
#define wstamp(a, cw, k) do { if ((a).trace && (threadIdx.x & 31) == 0) ctl->wclk[(cw)][(k)] = clock64(); } while (0)

// The abort flag as lane 0 of the warp sees it: a decision that guards warp-collective code (shuffles,
// reductions) must be the same in all 32 lanes, and the flag may change between two lanes' reads.
__device__ __forceinline__ bool warp_abort(const Ctl* ctl) { return __shfl_sync(FULL, ctl->abort, 0) != 0; }

__device__ __forceinline__ void set_error(const DecodeArgs& a, Ctl* ctl, uint32_t bit) {
  atomicOr(a.status, bit);
  ctl->abort = 1;
}


template <class SH, int TK>
__global__ void __launch_bounds__(DEC_THREADS, 1) k_decode(DecodeArgs a, int NS, int SS) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr SH L{};
  constexpr int H = SH::H, NCH = SH::NCH, LW = SH::LW, P = SH::P;
  constexpr int E = SH::E, K = SH::K, I = SH::I, Is = SH::Is;
  constexpr int NC = I / 16;                 // 16-column chunks of a routed h vector
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  const Smem sm = smem_map(L, T, G);
  uint4* xh = reinterpret_cast<uint4*>(smem + sm.xh);
  float2* xs = reinterpret_cast<float2*>(smem + sm.xs);
  float* hst = reinterpret_cast<float*>(smem + sm.hst);
  float* yv = reinterpret_cast<float*>(smem + sm.yv);
  float* shs = reinterpret_cast<float*>(smem + sm.shs);
  uint8_t* ring = smem + sm.ring;

  // per-CTA static ranges
  const int ra = range_lo(E + 1, cta, G), rb = range_lo(E + 1, cta + 1, G);       // router rows
  const int sa = range_lo(Is, cta, G), sbn = range_lo(Is, cta + 1, G);           // shared units
  const int r0 = range_lo(H, cta, G), r1 = range_lo(H, cta + 1, G);             // output rows
  const int nrow = r1 - r0;
  const int RPI = SS / (int)L.RR;                 // router rows per item
  const int SPI = (SS / (int)L.SU) & ~1;          // shared units per item (even)
  const int UPI = (SS / (int)L.EU) & ~1;          // expert units per item (even)
  const int SDPI = SS / (int)L.SDR;               // shared-down rows per item
  const int DRPI = SS / (int)L.DR;                // routed-down rows per stage
  // routed-down rows of EPI experts share a stage (expert j of the stage at row j * nrow); a warp reads eight
  // rows from the middle of an expert's rows on, so the last expert's reads must stay inside the stage
  const int EPI = nrow > 0 ? max(1, (DRPI - (nrow + 1) / 2 - 8) / nrow + 1) : 1;

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], NCW);
    }
    mbar_init(&ctl->route_ready, 1);
    ctl->abort = 0;
    if (a.trace) {
      for (int i = 0; i < 32; ++i) ctl->tclk[i] = 0;
      for (int i = 0; i < NCW * 4; ++i) ctl->wclk[i / 4][i % 4] = 0;
      ctl->tclk[30] = globaltimer();
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp(a, 0);
  // Programmatic dependent launch: the next kernel on the stream may be scheduled now (its CTAs take SMs as
  // this grid's CTAs leave and run their setup and weight copies), and it waits for this whole grid before
  // it touches global state.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
      const int U = ok ? ctl->U : 0;
#pragma unroll 1
      for (int sgi = 0; ok && sgi < nseg; ++sgi) {
        const int e = ctl->act_e[ctl->seg_a[sgi]], u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi];
        const uint8_t* gu = a.ex_gu + (size_t)e * L.exgu_expert;
#pragma unroll 1
        for (int u = u0; ok && u < u1; u += UPI)
          ok = issue(gu + (size_t)u * L.EU, (uint32_t)(min(UPI, u1 - u) * L.EU));
      }
      // the routed down rows, EPI experts a stage: one expect-tx for the stage, one copy per expert
#pragma unroll 1
      for (int aa0 = 0; ok && aa0 < U && nrow > 0; aa0 += EPI) {
        const int ne = min(EPI, U - aa0);
        const uint32_t eb = (uint32_t)(nrow * L.DR);
        if (ctl->abort) { ok = false; break; }
        if (n >= NS && !mbar_wait(&ctl->empty[ps], pph ^ 1u, a.timeout_ns)) {
          set_error(a, ctl, ERR_WAIT_EMPTY);
          ok = false;
          break;
        }
        mbar_expect_tx(&ctl->full[ps], eb * (uint32_t)ne);
#pragma unroll 1
        for (int j = 0; j < ne; ++j)
          bulk_g2s_hint(ring + (size_t)ps * SS + (size_t)j * eb,
                        a.ex_dn + (size_t)ctl->act_e[aa0 + j] * L.exdn_expert + (size_t)r0 * L.DR, eb,
                        &ctl->full[ps], pol);
        ++n;
        if (++ps == NS) { ps = 0; pph ^= 1u; }
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
    // the item i places after the next one (i = 0: the next one)
    auto stage_at = [&](int i) -> const uint8_t* {
      int s = cs + i;
      uint32_t ph = cph;
      while (s >= NS) { s -= NS; ph ^= 1u; }
      if (!ctl->abort && !mbar_wait(&ctl->full[s], ph, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_FULL);
      return ring + (size_t)s * SS;
    };
    auto acquire = [&]() -> const uint8_t* { return stage_at(0); };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[cs]);
      if (++cs == NS) { cs = 0; cph ^= 1u; }
    };

    // Everything the consumers read or write in global memory (x, logits, counters, hs, h, out) may belong to
    // the previous kernel on the stream until it has completed; the producer's weight copies above do not.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // ---- x prologue: (RMSNorm ->) fp16 activations in pair order, plus per-chunk pair-column sums; one
    // (token, 32-column chunk) item per consumer thread
    if (a.gamma) {
#pragma unroll 1
      for (int t = cw; t < T; t += NCW) {
        const uint16_t* xr = a.x + (size_t)t * H;
        float ss = 0.f;
#pragma unroll 1
        for (int i = lane * 8; i < H; i += 256) {
          const uint4 raw = __ldcg(reinterpret_cast<const uint4*>(xr + i));
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
    // one 8-column block per thread, the four blocks of a chunk on consecutive lanes
#pragma unroll 1
    for (int base = cw * 32; base < T * NCH * 4; base += CT) {
      const int i = base + lane, t = i / (NCH * 4), c = (i >> 2) % NCH, j = i & 3;
      const bool live = i < T * NCH * 4;
      float v[8];
      const uint4 raw = live ? __ldcg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H + c * 32 + j * 8)) : make_uint4(0, 0, 0, 0);
      const __half* h8 = reinterpret_cast<const __half*>(&raw);
      if (a.gamma) {
        const float rn = live ? ctl->rn[t] : 0.f;
        const uint4 graw = live ? *reinterpret_cast<const uint4*>(a.gamma + c * 32 + j * 8) : make_uint4(0, 0, 0, 0);
        const __half* g8 = reinterpret_cast<const __half*>(&graw);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __half2float(__float2half_rn(__half2float(h8[k]) * rn * __half2float(g8[k])));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __half2float(h8[k]);
      }
      quant_block8<LW, P>(v, live, t, c, j, xh, xs);
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 1);

    // ---- A1: router rows -> logits (a row per warp)
    for (int r = ra; r < rb; r += RPI) {
      const int nr = min(RPI, rb - r);
      const uint8_t* st = acquire();
      if (!warp_abort(ctl)) {
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
    // warps compute this CTA's shared-expert gate/up units; both join again before the routed gate/up.
    const int RW = T < 8 ? T : 8, AW = NCW - RW;
    if (cw < AW) {
      // ---- A2: shared-expert gate/up units, a pair per warp
#pragma unroll 1
      for (int u = sa; u < sbn; u += SPI) {
        const int nu = min(SPI, sbn - u);
        const uint8_t* st = acquire();
        if (!warp_abort(ctl)) {
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
      // this CTA's share of the routed units: segments of (active expert, unit range); then release the producer
      // The split is by work, not by units: active expert aa with n tokens weighs n per unit, so unit u of it
      // starts at work offset I * act_pb[aa] + u * n, and a CTA takes the units that start inside its slice of
      // the I * pairs total. With one token this is the plain split of the U * I units.
      auto plan = [&]() {
        const int U = ctl->U, W = I * (int)ctl->act_pb[U];
        const int lo = range_lo(W, cta, G), hi = range_lo(W, cta + 1, G);
        int nseg = 0;
#pragma unroll 1
        for (int aa = 0; aa < U && lo < hi; ++aa) {
          const int w0 = I * (int)ctl->act_pb[aa], n = (int)ctl->act_pb[aa + 1] - (int)ctl->act_pb[aa];
          if (w0 >= hi) break;
          if (w0 + I * n <= lo) continue;
          const int u0 = max(0, (lo - w0 + n - 1) / n), u1 = min(I, (hi - w0 + n - 1) / n);
          if (u0 >= u1) continue;
          if (nseg == DEC_MAXSEG) { set_error(a, ctl, ERR_SEGMENTS); break; }
          ctl->seg_a[nseg] = aa;
          ctl->seg_u0[nseg] = u0;
          ctl->seg_u1[nseg] = u1;
          ++nseg;
        }
        ctl->nseg = ctl->abort ? 0 : nseg;
        mbar_arrive(&ctl->route_ready);
        stamp(a, 5);
      };
      if (!warp_abort(ctl)) {
#pragma unroll 1
        for (int t = rt; t < T; t += RW) {
          const float* lg = a.logits + (size_t)t * (E + 1);
          int my_idx;
          float my_logit;
          warp_topk_lean<(E + 31) / 32, false>(lg, E, K, my_idx, my_logit);   // rows of E+1 floats: unaligned
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
      // bucketing: token masks per expert; active experts in ascending order with their first sorted pair
#pragma unroll 1
      for (int e = rtid; e < E; e += NT) ctl->emask[e] = 0u;
      named_bar(BAR_R, NT);
      if (!ctl->abort)
#pragma unroll 1
        for (int p = rtid; p < T * K; p += NT) atomicOr(&ctl->emask[ctl->ids[p / K][p % K]], 1u << (p / K));
      named_bar(BAR_R, NT);
      const int EPT = (E + NT - 1) / NT;
      int cnt = 0, pcnt = 0;
#pragma unroll 1
      for (int q = 0; q < EPT; ++q) {
        const int e = rtid * EPT + q;
        const uint32_t msk = e < E ? ctl->emask[e] : 0u;
        cnt += msk != 0u ? 1 : 0;
        pcnt += __popc(msk);
      }
      int incl = cnt, pincl = pcnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o), pv = __shfl_up_sync(FULL, pincl, o);
        if (lane >= o) { incl += v; pincl += pv; }
      }
      if (lane == 31) { ctl->warp_tot[rt] = incl; ctl->warp_tot2[rt] = pincl; }
      named_bar(BAR_R, NT);
      int base = 0, pbase = 0;
#pragma unroll 1
      for (int w = 0; w < rt; ++w) { base += ctl->warp_tot[w]; pbase += ctl->warp_tot2[w]; }
      int pos = base + incl - cnt, ppos = pbase + pincl - pcnt;
#pragma unroll 1
      for (int q = 0; q < EPT; ++q) {
        const int e = rtid * EPT + q;
        const uint32_t msk = e < E ? ctl->emask[e] : 0u;
        if (msk != 0u) {
          ctl->act_e[pos] = (uint16_t)e;
          ctl->act_mask[pos] = msk;
          ctl->act_pb[pos] = (uint16_t)ppos;
          ++pos;
          ppos += __popc(msk);
        }
      }
      if (rtid == NT - 1) {
        ctl->U = ctl->abort ? 0 : base + incl;
        ctl->act_pb[base + incl] = (uint16_t)(pbase + pincl);
      }
      named_bar(BAR_R, NT);
      if (rtid == 0) plan();
      // the sorted pairs: token and weight of each, and each token's pair per expert slot
      const int U = ctl->U;
#pragma unroll 1
      for (int aa = rtid; aa < U; aa += NT) {
        const int e = ctl->act_e[aa];
        uint32_t msk = ctl->act_mask[aa];
        int p = ctl->act_pb[aa];
#pragma unroll 1
        while (msk != 0u) {
          const int t = __ffs(msk) - 1;
          msk &= msk - 1u;
          ctl->pair_tok[p] = (uint8_t)t;
#pragma unroll 1
          for (int j = 0; j < K; ++j)
            if (ctl->ids[t][j] == e) {
              ctl->pair_w[p] = ctl->wts[t][j];
              ctl->tok_pair[t][j] = (uint8_t)p;
            }
          ++p;
        }
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

    // ---- C: the shared expert's down projection for this CTA's output rows (every CTA's hs); its weights came
    // in before routing, and it runs while the routed weights are still on their way
    if (ctid == 0 && !ctl->abort && !spin_geq(&a.counters[1], (uint32_t)G, a.timeout_ns))
      set_error(a, ctl, ERR_WAIT_HS);
    named_bar(BAR_C, CT);
    if (!ctl->abort)
#pragma unroll 1
      for (int i = ctid; i < T * Is / 4; i += CT)
        reinterpret_cast<float4*>(hst)[i] = __ldcg(reinterpret_cast<const float4*>(a.hs) + i);
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 9);
    // a row per warp; each lane holds 16 consecutive values of a token's hs as int16 with its own scale
#pragma unroll 1
    for (int r = r0; r < r1; r += SDPI) {
      const int nr = min(SDPI, r1 - r);
      const uint8_t* st = acquire();
      if (!warp_abort(ctl)) {
#pragma unroll 1
        for (int rr = cw; rr < nr; rr += NCW) {
          const uint8_t* row = st + (size_t)rr * L.SDR;
          const bool live = lane < Is / 16;
          const uint4 w = live ? *reinterpret_cast<const uint4*>(row + lane * 16) : make_uint4(0, 0, 0, 0);
          const float2 sb = live ? h2f(*reinterpret_cast<const uint32_t*>(row + Is + (lane >> 2) * 4)) : make_float2(0.f, 0.f);
#pragma unroll 1
          for (int tt = 0; tt < T; ++tt) {
            const float4* hv = reinterpret_cast<const float4*>(hst + (size_t)tt * Is + lane * 16);
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            const Act16 act = quant_lane16(live ? hv[0] : z4, live ? hv[1] : z4, live ? hv[2] : z4, live ? hv[3] : z4);
            const float rs = warp_sum(live ? down_int8(w, sb, act) : 0.f);
            if (lane == 0) shs[tt * nrow + (r + rr - r0)] = rs;
          }
        }
      }
      release();
    }
    if (ctid == 0) stamp(a, 10);

    // ---- B1: routed gate/up -> h of every (expert, token) pair, to global (row per sorted pair)
    const int nseg = ctl->nseg;
#pragma unroll 1
    for (int sgi = 0; sgi < nseg; ++sgi) {
      const int aa = ctl->seg_a[sgi], u0 = ctl->seg_u0[sgi], u1 = ctl->seg_u1[sgi];
      const int pb = ctl->act_pb[aa], ne = ctl->act_pb[aa + 1] - pb;
      const uint8_t* toks = ctl->pair_tok + pb;
      float* hrow = a.hbuf + (size_t)pb * I;
      if (sgi == 0) wstamp(a, cw, 0);
#pragma unroll 1
      for (int u = u0; u < u1; u += UPI) {
        const int nu = min(UPI, u1 - u);
        const uint8_t* st = acquire();
        if (!warp_abort(ctl)) {
          // pairs are numbered across the whole segment so that consecutive items go to different warps
          const int pbase = (u - u0) >> 1;
#pragma unroll 1
          for (int pr = (cw - pbase % NCW + NCW) % NCW; pr * 2 < nu; pr += NCW) {
            const uint8_t* ub = st + (size_t)(2 * pr) * L.EU;
            const int nvalid = (2 * pr + 1 < nu) ? 4 : 2;
            const int ui = u + 2 * pr;
#pragma unroll 1
            for (int tc = 0; tc < ne; tc += TK) {
              const int nt = min(TK, ne - tc);
              if (TK > 1 && nt == 1) {
                // a lone token (most experts at small batch under top-k routing): the single-token dot, not the
                // token-pair one with half of its products on a zero activation
                const DotR<4, 1> d1 = dot_rows<H, 4, 1, false>(ub, ub + H / 2, ub + L.EU, ub + L.EU + H / 2,
                                                               ub + H, ub + H + L.GB * 4, ub + L.EU + H,
                                                               ub + L.EU + H + L.GB * 4, nvalid, xh, xs, toks[tc],
                                                               toks[tc], 1);
                if (lane < 2) {
                  const float g = lane ? d1.v[0][2] : d1.v[0][0], up = lane ? d1.v[0][3] : d1.v[0][1];
                  if (2 * lane < nvalid) hrow[(size_t)tc * I + hpos<I>(ui + lane)] = silu_fast(g) * up;
                }
                continue;
              }
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
                if (tt < nt && 2 * k < nvalid) hrow[(size_t)(tc + tt) * I + hpos<I>(ui + k)] = silu_fast(g) * up;
              }
            }
          }
        }
        release();
      }
      if (sgi == 0) wstamp(a, cw, 1);
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) {
      stamp(a, 7);
      __threadfence();
      atomicAdd(&a.counters[2], 1u);
    }


    // ---- every CTA's routed h is in global memory
    if (ctid == 0 && !ctl->abort && !spin_geq(&a.counters[2], (uint32_t)G, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_H);
    if (ctid == 0) stamp(a, 11);
    named_bar(BAR_C, CT);   // thread 0's wait for every CTA's h precedes every read of it

    // ---- B2: routed down projection of this CTA's rows
    {
      const int U = ctl->U;
      // More tokens: every warp walks the active experts' down items in ring order. An expert's work is cut
      // into units of (half of this CTA's rows) x (up to PC of its token pairs), dealt round-robin to the
      // warps; a unit brings its pairs' h (lane-ordered rows of I floats) from L2 into registers and runs
      // eight rows as independent dot chains, one transposed reduction per pair.
      constexpr int PC = 2;
      const int half = (nrow + 1) / 2;
      int ui = 0;
      const uint8_t* stage = nullptr;
#pragma unroll 1
      for (int aa = 0; aa < U && nrow > 0; ++aa) {
        const int pb = ctl->act_pb[aa], na = (int)ctl->act_pb[aa + 1] - pb;
        const int nunits = 2 * ((na + PC - 1) / PC);
        if (aa % EPI == 0) stage = acquire();
        const uint8_t* item = stage + (size_t)(aa % EPI) * nrow * L.DR;
#pragma unroll 1
        for (int k = 0; k < nunits; ++k, ++ui) {
          if (ui % NCW != cw || warp_abort(ctl)) continue;
          const int rlo = (k & 1) ? half : 0, rhi = (k & 1) ? nrow : half;
          const int p0 = pb + (k >> 1) * PC, np = min(PC, pb + na - p0);
          // each pair's h: the lane's 16 values (lane order of the down dot) as int16 with the lane's scale
          const bool live = NC % 32 == 0 || lane < NC;
          Act16 act[PC];
#pragma unroll
          for (int pp = 0; pp < PC; ++pp) {
            const float4* hrow = reinterpret_cast<const float4*>(a.hbuf + (size_t)(p0 + pp) * I);
            const bool ok = live && pp < np;
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            act[pp] = quant_lane16(ok ? __ldcg(hrow + lane) : z4, ok ? __ldcg(hrow + NC + lane) : z4,
                                   ok ? __ldcg(hrow + 2 * NC + lane) : z4, ok ? __ldcg(hrow + 3 * NC + lane) : z4);
          }
          float v[PC][8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint8_t* row = item + (rlo + q) * (int)L.DR;
            const uint2 w = live ? *reinterpret_cast<const uint2*>(row + lane * 8) : make_uint2(0, 0);
            const float2 sb = live ? h2f(*reinterpret_cast<const uint32_t*>(row + I / 2 + (lane >> 2) * 4)) : make_float2(0.f, 0.f);
#pragma unroll
            for (int pp = 0; pp < PC; ++pp) v[pp][q] = live ? down_int4(w, sb, act[pp]) : 0.f;
          }
          const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
          const int idx = lane >> 2;
#pragma unroll
          for (int pp = 0; pp < PC; ++pp) {
            float x4[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const float keep = b4 ? v[pp][4 + kk] : v[pp][kk], give = b4 ? v[pp][kk] : v[pp][4 + kk];
              x4[kk] = keep + __shfl_xor_sync(FULL, give, 16);
            }
            float x2[2];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const float keep = b3 ? x4[2 + kk] : x4[kk], give = b3 ? x4[kk] : x4[2 + kk];
              x2[kk] = keep + __shfl_xor_sync(FULL, give, 8);
            }
            float z = (b2 ? x2[1] : x2[0]) + __shfl_xor_sync(FULL, b2 ? x2[0] : x2[1], 4);
            z += __shfl_xor_sync(FULL, z, 2);
            z += __shfl_xor_sync(FULL, z, 1);
            if ((lane & 3) == 0 && pp < np && rlo + idx < rhi) yv[(size_t)(p0 + pp) * nrow + rlo + idx] = z;
          }
        }
        if (aa % EPI == EPI - 1 || aa == U - 1) release();
      }
    }
    named_bar(BAR_C, CT);
    if (ctid == 0) stamp(a, 8);

    // ---- D: out = sum over the token's experts (fixed order) of w * y + sigmoid(g) * shared (+ residual)
    if (!ctl->abort)
#pragma unroll 1
      for (int i = ctid; i < T * nrow; i += CT) {
        const int t = i / nrow, rr = i % nrow;
        float acc = 0.f;
#pragma unroll 1
        for (int j = 0; j < K; ++j) acc += ctl->wts[t][j] * yv[(size_t)ctl->tok_pair[t][j] * nrow + rr];
        float v = acc + ctl->sg[t] * shs[t * nrow + rr];
        if (a.gamma) v += __half2float(__ushort_as_half(__ldcg(a.x + (size_t)t * H + r0 + rr)));
        const uint16_t o = __half_as_ushort(__float2half_rn(v));
        a.out[(size_t)t * H + r0 + rr] = o;
        if (a.out2) a.out2[(size_t)t * H + r0 + rr] = o;
      }
    named_bar(BAR_C, CT);
  }

  __syncthreads();
  if (a.trace) {
    if (threadIdx.x == 0) {
      stamp(a, 12);
      ctl->tclk[31] = globaltimer();
    }
    __syncthreads();
    if (threadIdx.x < 32) a.trace[cta * 32 + threadIdx.x] = ctl->tclk[threadIdx.x];
    else if (threadIdx.x < 32 + NCW * 4)
      a.trace[G * 32 + (cta * 16 + (threadIdx.x - 32) / 4) * 4 + (threadIdx.x - 32) % 4] =
          ctl->wclk[(threadIdx.x - 32) / 4][(threadIdx.x - 32) % 4];
  }
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

}  // namespace

size_t decode_hbuf_floats(const MoeLayout& L, int T) { return (size_t)T * L.K * L.I; }

bool decode_plan(const MoeLayout& L, int T, int grid, int max_smem, DecodeLaunch* out) {
  if (grid > DEC_MAXGRID || T < 1 || T > DEC_TMAX) return false;
  const int rows = (L.H + grid - 1) / grid;
  if (rows > DEC_MAXROWS) return false;
  DecodeLaunch pl;
  pl.grid = grid;
  pl.hp = 0;
  const Smem m = smem_map(L, T, grid);
  // 8 gate/up units (4 unit pairs, 4 warps) a stage: fewer, larger copies land the routed weights sooner.
  int SS = (int)(8 * L.EU);
  if (SS < 4 * L.H) SS = 4 * L.H;
  if ((int)(2 * L.SU) > SS) SS = (int)(2 * L.SU);
  if ((int)L.RR > SS) SS = (int)L.RR;
  if ((int)L.SDR > SS) SS = (int)L.SDR;
  if ((int)L.DR > SS) SS = (int)L.DR;
  SS = (SS + 127) & ~127;
  int NS = (max_smem - m.ring) / SS;
  if (NS > DEC_MAXNS) NS = DEC_MAXNS;
  if (NS < 4) return false;
  const int drpi = SS / (int)L.DR, dn_items = (rows + drpi - 1) / drpi;
  if (dn_items > NS / 2) return false;
  // every expert's rows are one stage, and a warp reads eight rows from the middle one on
  if ((rows + 1) / 2 + 8 > drpi || (rows + 1) / 2 > 8) return false;
  pl.NS = NS;
  pl.SS = SS;
  pl.smem = m.ring + NS * SS;
  *out = pl;
  return true;
}

std::mutex g_dec_attr_mutex;

// raise the dynamic shared-memory limit once per device and instantiation (the setting is per function and
// per device)
template <class SH, int TK>
static cudaError_t prepare_s(const DecodeLaunch& pl) {
  auto kern = k_decode<SH, TK>;
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dec_attr_mutex);
  if (configured[dev] < pl.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    configured[dev] = pl.smem > 232448 ? pl.smem : 232448;
  }
  return cudaSuccess;
}

template <class SH, int TK>
static cudaError_t launch_s(const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  auto kern = k_decode<SH, TK>;
  cudaError_t e = prepare_s<SH, TK>(pl);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(DEC_THREADS);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  // The grid-wide counters need every CTA resident at once: one CTA per SM (its shared memory admits no
  // second) and grid <= SM count guarantee it once the SMs are free. The launch is programmatic-dependent
  // rather than cooperative: a dependent grid can start only after every CTA of this one has run
  // launch_dependents, so it never holds an SM that a CTA of this grid still waits for.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, pl.NS, pl.SS);
}

template <class SH>
static bool is_shape(const MoeLayout& L) {
  return L.H == SH::H && L.E == SH::E && L.K == SH::K && L.I == SH::I && L.Is == SH::Is;
}

bool decode_supported(const MoeLayout& L) { return is_shape<ShapeProd>(L) || is_shape<ShapeTiny>(L); }

template <class SH>
static cudaError_t occupancy_s(const DecodeLaunch& pl, int* per_sm) {
  cudaError_t e = prepare_s<SH, 2>(pl);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, k_decode<SH, 2>, DEC_THREADS, pl.smem);
}

cudaError_t decode_occupancy(const MoeLayout& L, const DecodeLaunch& pl, int* ctas_per_sm) {
  if (is_shape<ShapeProd>(L)) return occupancy_s<ShapeProd>(pl, ctas_per_sm);
  if (is_shape<ShapeTiny>(L)) return occupancy_s<ShapeTiny>(pl, ctas_per_sm);
  return cudaErrorNotSupported;
}

cudaError_t decode_launch(const MoeLayout& L, const DecodeArgs& a, const DecodeLaunch& pl, cudaStream_t st) {
  if (is_shape<ShapeProd>(L)) return launch_s<ShapeProd, 2>(a, pl, st);
  if (is_shape<ShapeTiny>(L)) return launch_s<ShapeTiny, 2>(a, pl, st);
  return cudaErrorNotSupported;
}

}  // namespace moe
