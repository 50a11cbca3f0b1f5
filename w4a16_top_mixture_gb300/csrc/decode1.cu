// Fused single-token decode kernel of the W4A16 routed-MoE block (T = 1): one launch, one CTA per SM, every
// weight byte the token needs read from HBM exactly once.
//
// The kernel is built around two facts of a single-token call:
//   * A CTA's share of the call's weights (its router rows, shared-expert units and output rows, and its slice
//     of the eight selected experts) is about 120 KB at production width, so every copy lands in a region of
//     its own in shared memory: the producer never waits for a stage to be freed, and issues all the routed
//     copies at once as soon as the routing is known.
//   * The kernel needs at most ~113 KB of shared memory and a register budget that lets two CTAs share an SM.
//     The next call's CTAs (a programmatic-dependent launch) then become resident while this call still runs,
//     and load their router and shared-expert weights before this call ends.
//
// Roles: warp 0 is the producer (one lane issues 1-D bulk copies, each completing on an mbarrier of its own);
// warps 1..12 are consumers. In time order:
//   prologue  x (or RMSNorm(h) * gamma) -> fp16 activations in pair order, with per-chunk sums
//   A1        the CTA's router rows -> logits, each writer then adds its rows to a grid-wide count
//   A2        the CTA's shared-expert gate/up units -> hs, counted the same way
//   R         warp 0 waits for all E+1 logits, takes the top-k with the softmax weights and plans the CTA's
//             slice of the K*I routed units; the producer then issues the routed gate/up copies, and (once
//             the router and shared gate/up regions they overlay have been read) the routed down rows
//   C         two warps wait for all hs and run the shared expert's down projection of the CTA's output rows
//   B1        every warp takes unit pairs of the routed gate/up slice as they land (a shared work counter):
//             h = silu(Wg x) * (Wu x) to a global row per selected expert, counted grid-wide per unit
//   B2        once all K*I units are in, one bulk copy brings the K h vectors into shared memory; the routed
//             down projection of the CTA's output rows, a warp per (expert, half of the rows)
//   D         out = sum_j w_j y_j (selection order) + sigmoid(g) * shared (+ residual), one fp16 rounding
// Every wait is bounded; a timeout sets an error bit and the CTA drains its copies and leaves.
#include <cuda_fp16.h>
#include <mutex>
#include <stdint.h>

#include "decode.cuh"
#include "decode_dev.cuh"
#include "ptx.cuh"

// Where the CTAs allow the next launch on the stream to start (griddepcontrol.launch_dependents): 0 at the
// start, 1 once the routed gate/up copies are issued, 2 after the routed gate/up work, 3 after the routed down
// rows. At 2 the next launch's weight-only copies no longer compete with this launch's routed copies for HBM,
// and still land before this launch ends (12.7 against 13.2 us per step at 1).
#ifndef MOE_PDL_AT
#define MOE_PDL_AT 2
#endif
// routed gate/up units per bulk copy (even, so a unit pair never straddles two copies)
#ifndef MOE_PIECE_UNITS
#define MOE_PIECE_UNITS 8
#endif

namespace moe {

namespace {

constexpr int W1 = DEC1_NCW;
constexpr int CT1 = W1 * 32;
constexpr int BAR_ALL = 1;           // every consumer warp
constexpr int BAR_CT = 2;            // the shared-down team (two warps)
constexpr int BAR_A1 = 3;            // the two router warps
constexpr int MAXPIECE = 8;          // routed gate/up copies of one CTA
constexpr int PIECE_UNITS = MOE_PIECE_UNITS;
constexpr int A2W0 = 2;              // first warp of the shared gate/up work
constexpr int CTW0 = W1 - 2;         // first warp of the shared-down team

// The launch's one-shot mbarriers, one array: router rows / shared gate-up units / shared down rows landed
// (B_PRE + 0..2), routed gate/up copy i landed (B_GU + i), the CTA's rows of the j-th selected expert's down
// matrix landed (B_DN + j), routing and plan ready (B_ROUTE), every consumer warp done with the router and
// shared gate/up regions (B_RFREE), the routed h vectors landed (B_H).
enum : int { B_PRE = 0, B_GU = 3, B_DN = B_GU + MAXPIECE, B_ROUTE = B_DN + 16, B_RFREE, B_H, NBAR };
static_assert(NBAR <= 32, "armed barriers are tracked in a 32-bit mask");

struct Ctl1 {
  uint64_t bar[NBAR];
  volatile int abort;
  int next_pair;                     // shared work counter of B1
  int npiece, npair;
  int piece_slot[MAXPIECE];          // selected-expert slot of copy i
  int piece_u0[MAXPIECE], piece_u1[MAXPIECE];   // its units within the expert
  int piece_off[MAXPIECE];           // its byte offset in the gate/up region
  int piece_pair0[MAXPIECE + 1];     // its first unit pair (prefix over copies)
  int eid[16];                       // selected experts, selection order
  float wts[16];                     // their renormalised softmax weights
  float sg;                          // sigmoid of the shared-gate logit
  float rn;                          // 1 / RMS of the layer input (residual mode)
  float a1p[3][4];                   // the other router warps' parts of the router rows' dot products
  unsigned long long tclk[32];       // phase stamps (SM clock), flushed to the trace buffer at exit
  unsigned long long wclk[W1][4];
};
constexpr int CTL1_BYTES = (sizeof(Ctl1) + 127) & ~127;

struct Smem1 {   // byte offsets of the dynamic shared-memory regions, and the total
  int x16, xsc, yv, shs, sdn, dn, gu, total;
};

__host__ __device__ constexpr int al128(int v) { return (v + 127) & ~127; }
__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

// Regions: x16 the activations as int16 pairs and xsc their per-chunk (scale, sum) (see dot_rows); yv routed
// down results [slot][row]; shs shared down results [row]; sdn the shared down rows; dn the routed down rows
// [slot][rows], which first hold the router rows and the shared gate/up units (read before routing ends); gu the
// routed gate/up units, later the K routed h vectors.
template <class LT>
__host__ __device__ inline Smem1 smem1_map(const LT& L, int G) {
  Smem1 m;
  const int rows = cdiv(L.H, G), rmax = cdiv(L.E + 1, G), smax = cdiv(L.Is, G), umax = cdiv(L.K * L.I, G);
  const int half = (rows + 1) / 2, pad = half + 8 > rows ? half + 8 - rows : 0;   // B2 reads 8 rows a warp
  int o = CTL1_BYTES;
  m.x16 = o; o += al128(L.H * 2);
  m.xsc = o; o += al128(L.NCH * 8);
  m.yv = o;  o += al128(L.K * rows * 4);
  m.shs = o; o += al128(rows * 4);
  m.sdn = o; o += al128(rows * (int)L.SDR);
  m.dn = o;
  {
    const int dn = (L.K * rows + pad) * (int)L.DR, pre = rmax * (int)L.RR + smax * (int)L.SU;
    o += al128(dn > pre ? dn : pre);
  }
  m.gu = o;
  {
    const int gu = umax * (int)L.EU, hv = L.K * L.I * 4;
    o += al128(gu > hv ? gu : hv);
  }
  m.total = o;
  return m;
}

// Phase stamps (SM clock) exist only in the traced instantiation of the kernel (TR = true), so the untraced one
// carries none of their code.
#define stamp1(a, slot) do { if (TR) ctl->tclk[(slot)] = clock64(); } while (0)
#define wstamp1(a, cw, k) do { if (TR && (threadIdx.x & 31) == 0) ctl->wclk[(cw)][(k)] = clock64(); } while (0)

__device__ __forceinline__ void set_error1(const DecodeArgs& a, Ctl1* ctl, uint32_t bit) {
  atomicOr(a.status, bit);
  ctl->abort = 1;
}

// one bulk copy global -> shared completing on its own barrier (out of line: one copy of the code)
static __device__ __noinline__ void copy_in(uint64_t* bar, void* dst, const void* src, uint32_t bytes, uint64_t pol) {
  mbar_expect_tx(bar, bytes);
  bulk_g2s_hint(dst, src, bytes, bar, pol);
}

// bounded wait on a one-shot mbarrier (phase 0), skipped once the CTA is aborting
__device__ __forceinline__ void wait_landed(const DecodeArgs& a, Ctl1* ctl, uint64_t* bar) {
  if (!ctl->abort && !mbar_wait(bar, 0, a.timeout_ns)) set_error1(a, ctl, ERR_WAIT_FULL);
}

// The abort flag as lane 0 of the warp sees it: every decision that guards warp-collective code (shuffles,
// reductions) must be the same in all 32 lanes, and the flag may change between two lanes' reads.
__device__ __forceinline__ bool warp_abort(const Ctl1* ctl) {
  return __shfl_sync(FULL, ctl->abort, 0) != 0;
}

template <class SH, bool TR>
__global__ void __launch_bounds__(DEC1_THREADS, 2) k_decode1(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr SH L{};
  constexpr int H = SH::H, NCH = SH::NCH, LW = SH::LW;
  constexpr int E = SH::E, K = SH::K, I = SH::I, Is = SH::Is, GB = SH::GB;
  constexpr int NC = I / 16;                  // 16-column chunks of a routed h vector (one per lane)
  static_assert(NC <= 32 && Is / 16 <= 32, "a down row's columns must fit one warp, 16 a lane");
  const int G = gridDim.x, cta = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl1* ctl = reinterpret_cast<Ctl1*>(smem);
  const Smem1 sm = smem1_map(L, G);
  uint4* x16 = reinterpret_cast<uint4*>(smem + sm.x16);
  float2* xsc = reinterpret_cast<float2*>(smem + sm.xsc);
  float* yv = reinterpret_cast<float*>(smem + sm.yv);
  float* shs = reinterpret_cast<float*>(smem + sm.shs);
  uint8_t* sdn = smem + sm.sdn;
  uint8_t* dnr = smem + sm.dn;
  uint8_t* gur = smem + sm.gu;
  const float4* hst4 = reinterpret_cast<const float4*>(smem + sm.gu);

  const int rows_max = cdiv(H, G);
  const int rmax = cdiv(E + 1, G);
  const int ra = range_lo(E + 1, cta, G), rb = range_lo(E + 1, cta + 1, G);    // router rows
  const int sa = range_lo(Is, cta, G), sb = range_lo(Is, cta + 1, G);          // shared units
  const int r0 = range_lo(H, cta, G), r1 = range_lo(H, cta + 1, G);            // output rows
  const int nrow = r1 - r0;
  const int ulo = range_lo(K * I, cta, G), uhi = range_lo(K * I, cta + 1, G);  // routed units (slot-major)
  uint8_t* rtr = dnr;                                  // router rows, then the shared units, before routing
  uint8_t* sgu = dnr + (size_t)rmax * L.RR;

  if (threadIdx.x < NBAR) {
    mbar_init(&ctl->bar[threadIdx.x], threadIdx.x == B_RFREE ? W1 : 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    ctl->abort = 0;
    ctl->next_pair = 0;
    ctl->npiece = 0;
    ctl->npair = 0;
    if (TR) {
      for (int i = 0; i < 32; ++i) ctl->tclk[i] = 0;
      for (int i = 0; i < W1 * 4; ++i) ctl->wclk[i / 4][i % 4] = 0;
      ctl->tclk[30] = globaltimer();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp1(a, 0);
  if (MOE_PDL_AT == 0 && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t armed = 0;   // barriers with a copy in flight
      // weight-only copies: they depend on nothing the previous launch writes
      if (rb > ra) {
        copy_in(&ctl->bar[B_PRE], rtr, a.router + (size_t)ra * L.RR, (uint32_t)((rb - ra) * L.RR), pol);
        armed |= 1u << B_PRE;
      }
      if (sb > sa) {
        copy_in(&ctl->bar[B_PRE + 1], sgu, a.sh_gu + (size_t)sa * L.SU, (uint32_t)((sb - sa) * L.SU), pol);
        armed |= 1u << (B_PRE + 1);
      }
      if (nrow > 0) {
        copy_in(&ctl->bar[B_PRE + 2], sdn, a.sh_dn + (size_t)r0 * L.SDR, (uint32_t)(nrow * L.SDR), pol);
        armed |= 1u << (B_PRE + 2);
      }
      stamp1(a, 16);
      bool ok = mbar_wait(&ctl->bar[B_ROUTE], 0, a.timeout_ns * 4);
      if (!ok) set_error1(a, ctl, ERR_WAIT_ROUTE);
      if (ctl->abort) ok = false;
      stamp1(a, 17);
      // the routing warp has issued the routed gate/up copies (before its arrival); they are drained here too
      const int np = ok ? ctl->npiece : 0;
#pragma unroll 1
      for (int i = 0; i < np; ++i) armed |= 1u << (B_GU + i);
      if (MOE_PDL_AT == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      stamp1(a, 18);
      // the routed down rows overlay the router and shared gate/up regions: wait until every warp is done
      // with those
      if (ok && !mbar_wait(&ctl->bar[B_RFREE], 0, a.timeout_ns)) {
        set_error1(a, ctl, ERR_WAIT_EMPTY);
        ok = false;
      }
      const int nd = (ok && !ctl->abort && nrow > 0) ? K : 0;
#pragma unroll 1
      for (int j = 0; j < nd; ++j) {
        copy_in(&ctl->bar[B_DN + j], dnr + (size_t)j * rows_max * L.DR,
                a.ex_dn + (size_t)ctl->eid[j] * L.exdn_expert + (size_t)r0 * L.DR, (uint32_t)(nrow * L.DR), pol);
        armed |= 1u << (B_DN + j);
      }
      stamp1(a, 19);
      // drain: every issued copy must have landed before the CTA may leave
#pragma unroll 1
      for (uint32_t m = armed; m != 0u; m &= m - 1u)
        if (!mbar_wait(&ctl->bar[__ffs(m) - 1], 0, a.timeout_ns)) atomicOr(a.status, ERR_WAIT_FULL);
      stamp1(a, 20);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    // x, logits, counters, hs, h and out may belong to the previous launch until it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // this launch's epoch: the router logits are published tagged with it, and the exchange counts reach
    // ep * expected (CTA 0 of the previous launch advanced it). A launch that finds an earlier error still set
    // computes nothing: the counts and tags are consistent again only once the host has read and reset the
    // status.
    const uint32_t ep = __ldcg(a.counters + CNT_EPOCH) + 1u;
    uint64_t* cnt_hs = reinterpret_cast<uint64_t*>(a.counters + CNT_HS64);
    uint64_t* cnt_h = reinterpret_cast<uint64_t*>(a.counters + CNT_H64);
    if (__ldcg(a.status) != 0u && ctid == 0) {
      atomicOr(a.status, ERR_REFUSED);
      ctl->abort = 1;
    }
    if (ctid == 0) stamp1(a, 1);

    // ---- prologue: (RMSNorm ->) fp16 activations in pair order and per-chunk pair-column sums
    float rn = 1.f;
    if (a.gamma) {
      if (cw == 0) {
        float ss = 0.f;
#pragma unroll 1
        for (int i = lane * 8; i < H; i += 256) {
          const uint4 raw = __ldcg(reinterpret_cast<const uint4*>(a.x + i));
          const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(hv[k]);
            ss += f.x * f.x + f.y * f.y;
          }
        }
        ss = warp_sum(ss);
        if (lane == 0) ctl->rn = 1.0f / sqrtf(ss / (float)H + a.eps);
      }
      named_bar(BAR_ALL, CT1);
      rn = ctl->rn;
    }
    // one 8-column block per thread, the four blocks of a chunk on consecutive lanes
#pragma unroll 1
    for (int base = cw * 32; base < NCH * 4; base += CT1) {
      const int i = base + lane, c = i >> 2, j = i & 3;
      const bool live = i < NCH * 4;
      float v[8];
      const uint4 raw = live ? __ldcg(reinterpret_cast<const uint4*>(a.x + c * 32 + j * 8)) : make_uint4(0, 0, 0, 0);
      const __half* h8 = reinterpret_cast<const __half*>(&raw);
      if (a.gamma) {
        const uint4 graw = live ? *reinterpret_cast<const uint4*>(a.gamma + c * 32 + j * 8) : make_uint4(0, 0, 0, 0);
        const __half* g8 = reinterpret_cast<const __half*>(&graw);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __half2float(__float2half_rn(__half2float(h8[k]) * rn * __half2float(g8[k])));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __half2float(h8[k]);
      }
      quant_block8<LW, SH::P>(v, live, 0, c, j, x16, xsc);
    }
    named_bar(BAR_ALL, CT1);
    if (ctid == 0) stamp1(a, 2);

    // ---- A1: the CTA's router rows (at most four) -> logits, on warps that are idle until routing: A1W warps,
    // each half of a row set's chunks (with four warps, warps 0, 1 take rows 0 and 2 and warps 4, 5 rows 1 and
    // 3). Warps other than 0 hand their sums over in shared memory and warp 0 publishes them.
    {
      const int nr = rb - ra;
      constexpr int PR = (NCH + 31) / 32;            // chunk passes of a row (dot_rows' P)
#ifndef MOE_A1_WARPS
#define MOE_A1_WARPS 2
#endif
      constexpr int A1W = PR >= 2 ? MOE_A1_WARPS : 1;   // warps on the router rows
      static_assert(A1W == 1 || A1W == 2 || A1W == 4, "router warps");
      const int aw = cw < 2 ? cw : cw - 2;               // index among the router warps (cw 0, 1, 4, 5)
      const bool a1 = nr > 0 && (cw < (A1W < 2 ? A1W : 2) || (A1W == 4 && (cw == 4 || cw == 5)));
      if (a1) {
        wait_landed(a, ctl, &ctl->bar[B_PRE]);
        if (lane == 0 && cw == 0) stamp1(a, 27);
        const bool live = !warp_abort(ctl);
        DotR<4, 1> d = {};
        // this warp's rows: all of them with one or two warps; every other one with four (the pair index picks
        // the first), compacted to the front of the call
        const int pair = A1W == 4 ? aw >> 1 : 0, half = A1W == 1 ? 0 : (aw & 1);
        const int step = A1W == 4 ? 2 : 1;
        const int nv = A1W == 4 ? (nr - pair + 1) / 2 : nr;
        if (live && nv > 0) {
          const uint8_t* b0 = rtr + (size_t)min(pair, nr - 1) * L.RR;
          const uint8_t* b1 = rtr + (size_t)min(pair + step, nr - 1) * L.RR;
          const uint8_t* b2 = rtr + (size_t)min(pair + 2 * step, nr - 1) * L.RR;
          const uint8_t* b3 = rtr + (size_t)min(pair + 3 * step, nr - 1) * L.RR;
          d = dot_rows<H, 4, 1, true>(b0, b1, b2, b3, b0 + H, b1 + H, b2 + H, b3 + H, nv, x16, xsc, 0, 0, 1,
                                      half * PR / (A1W == 1 ? 1 : 2), (half + 1) * PR / (A1W == 1 ? 1 : 2));
        }
        if (A1W > 1) {
          // every router warp reaches the barrier whatever the abort flag says (it may change between reads)
          if (aw != 0 && lane == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) ctl->a1p[aw - 1][i] = d.v[0][i];
          }
          named_bar(BAR_A1, 32 * A1W);
          if (cw == 0) {
            // row pair * 1 + step * i of this warp's call i; with four warps warp 0 holds rows 0, 2 and the
            // pair-1 warps rows 1, 3
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = 0.f;
            if (A1W == 2) {
#pragma unroll
              for (int i = 0; i < 4; ++i) v[i] = d.v[0][i] + ctl->a1p[0][i];
            } else {
              v[0] = d.v[0][0] + ctl->a1p[0][0];
              v[2] = d.v[0][1] + ctl->a1p[0][1];
              v[1] = ctl->a1p[1][0] + ctl->a1p[2][0];
              v[3] = ctl->a1p[1][1] + ctl->a1p[2][1];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) d.v[0][i] = v[i];
          }
        }
        if (cw == 0 && live) {
          if (lane == 0) stamp1(a, 28);
          // one {logit, epoch} word per row and copy: a reader that sees the tag has the value. Lane c writes
          // copy c (test hook: CTA 0 never publishes, so every reader's bounded wait runs out)
          if (lane < XLOG_COPIES && !(a.skip_arrive && ra == 0)) {
            uint64_t* dst = a.xlog + (size_t)lane * xlog_stride(E) + ra;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (i < nr) st_relaxed_u64(dst + i, ((uint64_t)ep << 32) | __float_as_uint(d.v[0][i]));
          }
          if (lane == 0) stamp1(a, 25);
        }
      }
    }
    // ---- A2: shared-expert gate/up units -> hs, a unit pair per warp
    {
      const int nsu = sb - sa, nsp = (nsu + 1) / 2;
      if (cw >= A2W0 && cw - A2W0 < nsp) {
        wait_landed(a, ctl, &ctl->bar[B_PRE + 1]);
        int done = 0;
        if (!warp_abort(ctl)) {
#pragma unroll 1
          for (int pr = cw - A2W0; pr < nsp; pr += W1 - A2W0) {
            const uint8_t* ub = sgu + (size_t)(2 * pr) * L.SU;
            const int nu = min(2, nsu - 2 * pr);
            const DotR<4, 1> d = dot_rows<H, 4, 1, true>(ub, ub + H, ub + L.SU, ub + L.SU + H, ub + 2 * H,
                                                         ub + 2 * H + GB * 4, ub + L.SU + 2 * H,
                                                         ub + L.SU + 2 * H + GB * 4, 2 * nu, x16, xsc, 0, 0, 1);
            if (lane < nu) {
              const float g = lane ? d.v[0][2] : d.v[0][0], up = lane ? d.v[0][3] : d.v[0][1];
              a.hs[sa + 2 * pr + lane] = silu_fast(g) * up;
            }
            done += nu;
          }
        }
        __syncwarp();
        if (lane == 0 && done > 0) red_release_add_u64(cnt_hs, (uint64_t)done);
      }
    }
    // this warp no longer reads the router or shared gate/up regions
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->bar[B_RFREE]);

    // ---- R: routing (warp 0): all E+1 logits -> top-k, softmax weights, sigmoid gate, the CTA's plan; the warp
    // issues the CTA's routed gate/up copies itself, one lane per copy
    if (cw == 0) {
      constexpr int EPL = (E + 31) / 32;
      // poll the tagged logits until every one carries this launch's epoch; lane l holds experts l*EPL..,
      // lane 0 also the shared-expert gate logit (row E). Each CTA polls one of the copies, so that the 152
      // readers do not all queue on the same few cache lines.
      uint32_t key[EPL];
      float gl = 0.f;
      bool got = false;
      const uint64_t* xl = a.xlog + (size_t)(cta % XLOG_COPIES) * xlog_stride(E);
      if (!warp_abort(ctl)) {
        const uint64_t t0 = globaltimer();
#pragma unroll 1
        for (int round = 0;; ++round) {
#ifndef MOE_POLL_NS
#define MOE_POLL_NS 64
#endif
          if (MOE_POLL_NS > 0 && round > 0) __nanosleep(MOE_POLL_NS);
          bool fresh = true;
          if (E % 64 == 0 && EPL % 2 == 0) {
#pragma unroll
            for (int i = 0; i < EPL; i += 2) {
              uint64_t w0, w1;
              ld_relaxed_u64x2(xl + lane * EPL + i, w0, w1);
              fresh = fresh && (uint32_t)(w0 >> 32) == ep && (uint32_t)(w1 >> 32) == ep;
              key[i] = topk_key(__uint_as_float((uint32_t)w0));
              key[i + 1] = topk_key(__uint_as_float((uint32_t)w1));
            }
          } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
              const int e = lane * EPL + i;
              const uint64_t w = e < E ? ld_relaxed_u64(xl + e) : ((uint64_t)ep << 32);
              fresh = fresh && (uint32_t)(w >> 32) == ep;
              key[i] = e < E ? topk_key(__uint_as_float((uint32_t)w)) : 0u;
            }
          }
          if (lane == 0) {
            const uint64_t w = ld_relaxed_u64(xl + E);
            fresh = fresh && (uint32_t)(w >> 32) == ep;
            gl = __uint_as_float((uint32_t)w);
          }
          if (__all_sync(FULL, fresh)) { got = true; break; }
          if (__shfl_sync(FULL, globaltimer() - t0 > a.timeout_ns || ctl->abort ? 1 : 0, 0)) break;
        }
        if (!got && lane == 0) set_error1(a, ctl, ERR_WAIT_LOGITS);
        // every CTA read the epoch before it published its rows, so once all rows carry it the next launch's
        // epoch can be set: the next launch reads it only after this one has completed
        if (got && cta == 0 && lane == 0) a.counters[CNT_EPOCH] = ep;
      }
      __syncwarp();
      if (lane == 0) stamp1(a, 3);
      // CTA 0 records the logits (the top-k consumes the keys)
      if (cta == 0 && a.rec_ids) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (lane * EPL + i < E) a.logits[lane * EPL + i] = topk_logit(key[i]);
        if (lane == 0) a.logits[E] = gl;
      }
      int my_idx = 0;
      uint32_t my_key = 0;
      if (got) warp_topk_keys<EPL>(key, K, my_idx, my_key);
      // the CTA's slice [ulo, uhi) of the K*I routed units (slot-major) in copies of at most PIECE_UNITS units
      // inside one expert: the slice covers at most two experts (the plan checks it), so copy k is, in closed
      // form, the k-th PIECE_UNITS-step of the first expert's part or then of the second's. The copies need only
      // the selected experts: they go out first, the softmax weights (read at the very end) after them.
      {
        const int js = ulo / I, cut = min(uhi, (js + 1) * I);
        const int n0 = cdiv(cut - ulo, PIECE_UNITS), n1 = cdiv(uhi - cut, PIECE_UNITS);
        const int np = !got || warp_abort(ctl) || uhi <= ulo ? 0 : n0 + n1;
        const bool first = lane < n0;
        const int b0 = first ? ulo : cut, k = first ? lane : lane - n0;
        const int u = b0 + k * PIECE_UNITS, u1 = min(first ? cut : uhi, u + PIECE_UNITS);
        const int j = lane < np ? u / I : 0;
        const int e = __shfl_sync(FULL, my_idx, j);   // the expert in selection slot j
        if (lane < np)
          copy_in(&ctl->bar[B_GU + lane], gur + (u - ulo) * (int)L.EU,
                  a.ex_gu + (size_t)e * L.exgu_expert + (size_t)(u - j * I) * L.EU, (uint32_t)((u1 - u) * L.EU),
                  policy_evict_first());
        if (lane < np) {
          ctl->piece_slot[lane] = j;
          ctl->piece_u0[lane] = u - j * I;
          ctl->piece_u1[lane] = u1 - j * I;
          ctl->piece_off[lane] = (u - ulo) * (int)L.EU;
          // unit pairs before this copy: whole first-part copies hold PIECE_UNITS / 2 pairs each
          ctl->piece_pair0[lane] = first ? k * (PIECE_UNITS / 2) : cdiv(cut - ulo, 2) + k * (PIECE_UNITS / 2);
        }
        if (lane < K) ctl->eid[lane] = my_idx;
        if (lane == 0) {
          ctl->piece_pair0[np] = np == 0 ? 0 : cdiv(cut - ulo, 2) + cdiv(uhi - cut, 2);
          ctl->npiece = np;
          ctl->npair = np == 0 ? 0 : cdiv(cut - ulo, 2) + cdiv(uhi - cut, 2);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->bar[B_ROUTE]);
          stamp1(a, 4);
        }
      }
      // softmax over the selected logits (selection order), the shared expert's sigmoid gate
      const float my_logit = topk_logit(my_key);
      const float mx = __shfl_sync(FULL, my_logit, 0);
      if (lane == 0) stamp1(a, 21);
      const float ex = lane < K ? __expf(my_logit - mx) : 0.f;
      const float Z = warp_sum(ex);
      const float wv = __fdividef(ex, Z);
      if (lane == 0) stamp1(a, 22);
      if (lane < K) ctl->wts[lane] = wv;
      if (lane == 0) ctl->sg = __frcp_rn(1.0f + __expf(-gl));
      // CTA 0's routing record (selection order; moe_block_debug_last_routing sorts it)
      if (cta == 0 && a.rec_ids) {
        if (lane < K) {
          a.rec_ids[lane] = my_idx;
          a.rec_w[lane] = wv;
        }
        if (lane == 0 && a.rec_sg) a.rec_sg[0] = ctl->sg;
      }
    }

    // ---- C: the shared expert's down projection of the CTA's rows (two warps, off the critical path); every
    // lane holds 16 consecutive values of hs as int16 with its own scale
    if (cw >= CTW0) {
      const int ct = ctid - CTW0 * 32;
      if (ct == 0) stamp1(a, 23);
      if (ct == 0 && !ctl->abort && !spin_geq_u64(cnt_hs, (uint64_t)ep * Is, a.timeout_ns))
        set_error1(a, ctl, ERR_WAIT_HS);
      named_bar(BAR_CT, 64);
      if (nrow > 0) wait_landed(a, ctl, &ctl->bar[B_PRE + 2]);
      if (!warp_abort(ctl)) {
        constexpr int NCS = Is / 16;             // lanes holding hs values
        float4 hv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          hv[j] = lane < NCS ? __ldcg(reinterpret_cast<const float4*>(a.hs) + lane * 4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        const Act16 act = quant_lane16(hv[0], hv[1], hv[2], hv[3]);
#pragma unroll 1
        for (int rr = cw - CTW0; rr < nrow; rr += W1 - CTW0) {
          const uint8_t* row = sdn + (size_t)rr * L.SDR;
          float rs = 0.f;
          if (lane < NCS) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + lane * 16);
            const float2 sbp = h2f(*reinterpret_cast<const uint32_t*>(row + Is + (lane >> 2) * 4));
            rs = down_int8(w, sbp, act);
          }
          rs = warp_sum(rs);
          if (lane == 0) shs[rr] = rs;
        }
      }
      if (ct == 0) stamp1(a, 24);
    }

    // ---- B1: routed gate/up unit pairs as they land -> h rows in global memory
    if (!ctl->abort && !mbar_wait(&ctl->bar[B_ROUTE], 0, a.timeout_ns * 4)) set_error1(a, ctl, ERR_WAIT_ROUTE);
    {
      const int npair = ctl->npair;
      int done = 0;
#pragma unroll 1
      while (true) {
        int q = 0;
        if (lane == 0) q = atomicAdd(&ctl->next_pair, 1);
        q = __shfl_sync(FULL, q, 0);
        if (q >= npair || warp_abort(ctl)) break;
        int pc = 0;
        while (ctl->piece_pair0[pc + 1] <= q) ++pc;
        const int pp = q - ctl->piece_pair0[pc];
        const int u0 = ctl->piece_u0[pc] + 2 * pp, nu = min(2, ctl->piece_u1[pc] - u0);
        wait_landed(a, ctl, &ctl->bar[B_GU + pc]);
        if (warp_abort(ctl)) break;
        const uint8_t* ub = gur + ctl->piece_off[pc] + (size_t)(2 * pp) * L.EU;
        const DotR<4, 1> d = dot_rows<H, 4, 1, false>(ub, ub + H / 2, ub + L.EU, ub + L.EU + H / 2, ub + H,
                                                      ub + H + GB * 4, ub + L.EU + H, ub + L.EU + H + GB * 4,
                                                      2 * nu, x16, xsc, 0, 0, 1);
        if (lane < nu) {
          const float g = lane ? d.v[0][2] : d.v[0][0], up = lane ? d.v[0][3] : d.v[0][1];
          a.hbuf[(size_t)ctl->piece_slot[pc] * I + hpos<I>(u0 + lane)] = silu_fast(g) * up;
        }
        done += nu;
      }
      __syncwarp();
      if (lane == 0 && done > 0) red_release_add_u64(cnt_h, (uint64_t)done);
      wstamp1(a, cw, 1);
    }
    named_bar(BAR_ALL, CT1);   // the CTA's gate/up region is no longer read
    if (ctid == 0) {
      stamp1(a, 5);
      if (MOE_PDL_AT == 2) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      if (!ctl->abort && !spin_geq_u64(cnt_h, (uint64_t)ep * (K * I), a.timeout_ns)) set_error1(a, ctl, ERR_WAIT_H);
      stamp1(a, 6);
      if (!ctl->abort) {
        fence_proxy_async_global();
        mbar_expect_tx(&ctl->bar[B_H], (uint32_t)(K * I * 4));
        bulk_g2s(gur, a.hbuf, (uint32_t)(K * I * 4), &ctl->bar[B_H]);
      } else {
        mbar_arrive(&ctl->bar[B_H]);
      }
    }
    if (!ctl->abort && !mbar_wait(&ctl->bar[B_H], 0, a.timeout_ns)) set_error1(a, ctl, ERR_WAIT_FULL);
    if (ctid == 0) stamp1(a, 7);
    wstamp1(a, cw, 2);

    // ---- B2: routed down projection of the CTA's rows: a warp per (selected expert, half of the rows), h in
    // registers, eight rows as independent chains (rows past the half are read and dropped), one transposed
    // reduction per eight rows
    {
      const int half = (nrow + 1) / 2;
#pragma unroll 1
      for (int wi = cw; wi < 2 * K && !warp_abort(ctl); wi += W1) {
        const int j = wi >> 1, rlo = (wi & 1) ? half : 0, rhi = (wi & 1) ? nrow : half;
        if (rlo >= rhi) continue;
        wait_landed(a, ctl, &ctl->bar[B_DN + j]);
        if (warp_abort(ctl)) break;
        // the lane's 16 values of h_j (lane order of the down dot) as int16 with the lane's own scale
        const bool live = NC % 32 == 0 || lane < NC;
        float4 hv[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) hv[jj] = live ? hst4[(size_t)j * 4 * NC + jj * NC + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        const Act16 act = quant_lane16(hv[0], hv[1], hv[2], hv[3]);
        if (wi == cw) wstamp1(a, cw, 0);
        const uint8_t* item0 = dnr + (size_t)j * rows_max * L.DR;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint8_t* row = item0 + (rlo + q) * (int)L.DR;
          v[q] = live ? down_int4(*reinterpret_cast<const uint2*>(row + lane * 8),
                                  h2f(*reinterpret_cast<const uint32_t*>(row + I / 2 + (lane >> 2) * 4)), act)
                      : 0.f;
        }
        // transposed reduction of the eight values over the warp: lane 4i ends with row rlo + i
        const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
        float x4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float keep = b4 ? v[4 + k] : v[k], give = b4 ? v[k] : v[4 + k];
          x4[k] = keep + __shfl_xor_sync(FULL, give, 16);
        }
        float x2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float keep = b3 ? x4[2 + k] : x4[k], give = b3 ? x4[k] : x4[2 + k];
          x2[k] = keep + __shfl_xor_sync(FULL, give, 8);
        }
        float z = (b2 ? x2[1] : x2[0]) + __shfl_xor_sync(FULL, b2 ? x2[0] : x2[1], 4);
        z += __shfl_xor_sync(FULL, z, 2);
        z += __shfl_xor_sync(FULL, z, 1);
        const int idx = lane >> 2;
        if ((lane & 3) == 0 && rlo + idx < rhi) yv[j * rows_max + rlo + idx] = z;
      }
      wstamp1(a, cw, 3);
    }
    named_bar(BAR_ALL, CT1);
    if (ctid == 0) stamp1(a, 8);
    if (MOE_PDL_AT == 3 && ctid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- D: out = sum_j w_j y_j (selection order) + sigmoid(g) * shared row (+ residual), one fp16 rounding
    if (!ctl->abort) {
#pragma unroll 1
      for (int rr = ctid; rr < nrow; rr += CT1) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) acc += ctl->wts[j] * yv[j * rows_max + rr];
        float v = acc + ctl->sg * shs[rr];
        if (a.gamma) v += __half2float(__ushort_as_half(__ldcg(a.x + r0 + rr)));
        const uint16_t o = __half_as_ushort(__float2half_rn(v));
        a.out[r0 + rr] = o;
        if (a.out2) a.out2[r0 + rr] = o;
      }
    }
  }

  __syncthreads();
  if (TR) {
    if (threadIdx.x == 0) {
      stamp1(a, 12);
      ctl->tclk[31] = globaltimer();
    }
    __syncthreads();
    if (threadIdx.x < 32) a.trace[cta * 32 + threadIdx.x] = ctl->tclk[threadIdx.x];
    else if (threadIdx.x < 32 + W1 * 4)
      a.trace[G * 32 + (cta * 16 + (threadIdx.x - 32) / 4) * 4 + (threadIdx.x - 32) % 4] =
          ctl->wclk[(threadIdx.x - 32) / 4][(threadIdx.x - 32) % 4];
  }
}

template <class SH>
static bool is_shape1(const MoeLayout& L) {
  return L.H == SH::H && L.E == SH::E && L.K == SH::K && L.I == SH::I && L.Is == SH::Is;
}

// per-device, per-kernel: the dynamic shared-memory limit the kernel has been given (0 = not yet)
std::mutex g_attr_mutex;
int g_attr_smem[4][64];

// the kernel's shared-memory attributes on the current device (once per device and instantiation)
template <class SH, int KID>
static cudaError_t prepare1(bool tr, const Decode1Launch& pl) {
  auto kern = tr ? k_decode1<SH, true> : k_decode1<SH, false>;
  const int kid = KID * 2 + (tr ? 1 : 0);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_attr_mutex);
  if (g_attr_smem[kid][dev] < pl.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    // the whole unified L1/shared array as shared memory, so that two CTAs fit on one SM
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    g_attr_smem[kid][dev] = pl.smem;
  }
  return cudaSuccess;
}

template <class SH, int KID>
static cudaError_t occupancy1(const Decode1Launch& pl, int* per_sm) {
  cudaError_t e = prepare1<SH, KID>(false, pl);
  if (e == cudaSuccess) e = prepare1<SH, KID>(true, pl);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, k_decode1<SH, false>, DEC1_THREADS, pl.smem);
}

template <class SH, int KID>
static cudaError_t launch1(const DecodeArgs& a, const Decode1Launch& pl, cudaStream_t st) {
  const bool tr = a.trace != nullptr;
  auto kern = tr ? k_decode1<SH, true> : k_decode1<SH, false>;
  cudaError_t e = prepare1<SH, KID>(tr, pl);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(DEC1_THREADS);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class SH>
static bool plan1_s(const MoeLayout& L, int grid, int max_smem, Decode1Launch* out) {
  constexpr SH S{};
  if (grid < 1 || grid > DEC_MAXGRID) return false;
  const Smem1 m = smem1_map(S, grid);
  if (m.total > max_smem) return false;
  const int rows = cdiv(S.H, grid), umax = cdiv(S.K * S.I, grid);
  if ((rows + 1) / 2 > 8) return false;                                  // B2: eight rows a warp
  // a CTA's slice of the routed units spans at most two experts, in copies of PIECE_UNITS units
  if (umax > S.I || cdiv(umax, PIECE_UNITS) + 1 > MAXPIECE) return false;
  out->grid = grid;
  out->smem = m.total;
  // two CTAs of 1 KB reserved shared memory each on an SM of 228 KB
  out->two_per_sm = 2 * (m.total + 1024) <= 233472 ? 1 : 0;
  (void)L;
  return true;
}

}  // namespace

bool decode1_plan(const MoeLayout& L, int grid, int max_smem, Decode1Launch* out) {
  if (is_shape1<ShapeProd>(L)) return plan1_s<ShapeProd>(L, grid, max_smem, out);
  if (is_shape1<ShapeTiny>(L)) return plan1_s<ShapeTiny>(L, grid, max_smem, out);
  return false;
}

cudaError_t decode1_occupancy(const MoeLayout& L, const Decode1Launch& pl, int* ctas_per_sm) {
  if (is_shape1<ShapeProd>(L)) return occupancy1<ShapeProd, 0>(pl, ctas_per_sm);
  if (is_shape1<ShapeTiny>(L)) return occupancy1<ShapeTiny, 1>(pl, ctas_per_sm);
  return cudaErrorNotSupported;
}

cudaError_t decode1_launch(const MoeLayout& L, const DecodeArgs& a, const Decode1Launch& pl, cudaStream_t st) {
  if (is_shape1<ShapeProd>(L)) return launch1<ShapeProd, 0>(a, pl, st);
  if (is_shape1<ShapeTiny>(L)) return launch1<ShapeTiny, 1>(a, pl, st);
  return cudaErrorNotSupported;
}

}  // namespace moe
