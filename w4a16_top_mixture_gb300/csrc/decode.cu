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
constexpr int PMAX = DEC_TMAX * 16;   // (token, expert) pairs

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
  static constexpr size_t DR = c_align16((size_t)I / 2 + (size_t)GI * 4);
  static constexpr size_t exgu_expert = (size_t)I * EU;
  static constexpr size_t exdn_expert = (size_t)H * DR;
};
using ShapeProd = Shape<2048, 256, 8, 512, 512>;
using ShapeTiny = Shape<512, 32, 4, 128, 128>;

struct Ctl {
  uint64_t full[DEC_MAXNS];
  uint64_t empty[DEC_MAXNS];
  uint64_t route_ready;
  uint64_t hbar;                      // the routed h of a single-token launch has landed in shared memory
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
  int xh, xs, hss, hst, yv, shs, ring;
};

// xh: x as fp16 [T][P][4 blocks][LW lanes] uint4 (the 8 columns of a block in pair order 0 4 1 5 2 6 3 7);
// xs: per (token, 32-column chunk) the sums of x over the chunk's "low" and "high" pair columns;
// hss: 16-column sums of the shared expert's hs; hst: phase C's hs [T][Is], then (one token) the routed h
// of the K pairs, bulk-copied in the lane order of the down dot; yv: routed down results [pair][row];
// shs: shared down results [token][row]; ring: the weight stages.
template <class LT>
__host__ __device__ inline Smem smem_map(const LT& L, int T, int grid, int hp) {
  Smem m;
  const int rows = (L.H + grid - 1) / grid;
  int o = CTL_BYTES;
  m.xh = o;   o += (T * L.H * 2 + 127) & ~127;
  m.xs = o;   o += (T * L.NCH * 8 + 127) & ~127;
  m.hss = o;  o += (T * (L.Is / 16) * 4 + 127) & ~127;
  m.hst = o;
  {
    const int f = hp * L.I > T * L.Is ? hp * L.I : T * L.Is;
    o += (f * 4 + 127) & ~127;
  }
  m.yv = o;   o += (T * L.K * rows * 4 + 127) & ~127;
  m.shs = o;  o += (T * rows * 4 + 127) & ~127;
  m.ring = o;
  return m;
}

__device__ __forceinline__ int range_lo(int n, int c, int G) { return (int)(((unsigned)n * (unsigned)c) / (unsigned)G); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Phase stamps read the SM clock into shared memory (a few cycles, so tracing barely perturbs the kernel) and
// are written out once at exit: trace[cta*32 + slot] (slots 30 / 31: globaltimer at start / end, which place
// the CTA's clock on a common time axis) and per-warp stamps trace[grid*32 + (cta*16 + warp)*4 + k].
#define stamp(a, slot) do { if ((a).trace) ctl->tclk[(slot)] = clock64(); } while (0)
#define wstamp(a, cw, k) do { if ((a).trace && (threadIdx.x & 31) == 0) ctl->wclk[(cw)][(k)] = clock64(); } while (0)

__device__ __forceinline__ void set_error(const DecodeArgs& a, Ctl* ctl, uint32_t bit) {
  atomicOr(a.status, bit);
  ctl->abort = 1;
}

template <int NR, int TK>
struct DotR {
  float v[TK][NR];
};

// Routed h vectors are stored in the lane order of the down dot: unit u = 16 c + 4 j + m (lane chunk c,
// float4 j, component m) sits at float index (j * (I/16) + c) * 4 + m, so that a linear copy of a vector into
// shared memory lets lane c read its float4 j at consecutive 16-byte addresses across the warp.
template <int I>
__device__ __forceinline__ int hpos(int u) {
  return (((u & 15) >> 2) * (I / 16) + (u >> 4)) * 4 + (u & 3);
}

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
// Once the k experts are known, lane j asks L2 to prefetch the weights of the j-th one that this CTA's share
// of the work is likely to read: a 1/G slice of its gate/up block (the grid as a whole covers the expert) and
// this CTA's own rows of its down matrix.
template <int EPL>
__device__ __noinline__ void warp_topk(const float* __restrict__ lg, int E, int K, int lane, int& my_idx,
                                       float& my_logit, const uint8_t* pf_gu, size_t pf_gu_sz,
                                       const uint8_t* pf_dn, size_t pf_dn_sz, size_t dn0, size_t dn1) {
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
  if (lane < K && pf_gu) {
    if (gu1 > gu0) prefetch_l2(pf_gu + (size_t)my_idx * pf_gu_sz + gu0, (uint32_t)(gu1 - gu0));
    if (dn1 > dn0) prefetch_l2(pf_dn + (size_t)my_idx * pf_dn_sz + dn0, (uint32_t)(dn1 - dn0));
  }
  const uint32_t b = (my_key & 0x80000000u) ? (my_key & 0x7FFFFFFFu) : ~my_key;
  my_logit = __uint_as_float(b);
}

template <class SH, int TK>
__global__ void __launch_bounds__(DEC_THREADS, 1) k_decode(DecodeArgs a, int NS, int SS, int hp) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr SH L{};
  constexpr int H = SH::H, NCH = SH::NCH, LW = SH::LW, P = SH::P;
  constexpr int E = SH::E, K = SH::K, I = SH::I, Is = SH::Is;
  constexpr int NC = I / 16;                 // 16-column chunks of a routed h vector
  constexpr bool ONE = TK == 1;              // single-token launch (T == 1)
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  const Smem sm = smem_map(L, T, G, hp);
  uint4* xh = reinterpret_cast<uint4*>(smem + sm.xh);
  float2* xs = reinterpret_cast<float2*>(smem + sm.xs);
  float* hss = reinterpret_cast<float*>(smem + sm.hss);
  float* hst = reinterpret_cast<float*>(smem + sm.hst);
  float4* hst4 = reinterpret_cast<float4*>(smem + sm.hst);
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
  const int DRPI = SS / (int)L.DR;                // routed-down rows per item
  const int dn_items = (nrow + DRPI - 1) / DRPI;  // routed-down items per active expert

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], NCW);
    }
    mbar_init(&ctl->route_ready, 1);
    mbar_init(&ctl->hbar, 1);
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
#pragma unroll 1
      for (int aa = 0; ok && aa < U; ++aa) {
        const uint8_t* dn = a.ex_dn + (size_t)ctl->act_e[aa] * L.exdn_expert + (size_t)r0 * L.DR;
#pragma unroll 1
        for (int rr = 0; ok && rr < nrow; rr += DRPI)
          ok = issue(dn + (size_t)rr * L.DR, (uint32_t)(min(DRPI, nrow - rr) * L.DR));
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
    // warps compute this CTA's shared-expert gate/up units; both join again before the routed gate/up.
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
      // No L2 prefetch: its copy-engine requests (two per selected expert and token) queue ahead of, and
      // delay, the weight copies the producer issues right after routing.
      const uint8_t* pf_gu = nullptr;
      const size_t dn0 = (size_t)r0 * L.DR, dn1 = (size_t)r1 * L.DR;
      if (ONE) {
        // one token: the K experts in selection order are the active experts, one pair each
        const float* lg = a.logits;
        int my_idx = 0;
        float my_logit = 0.f;
        if (!ctl->abort)
          warp_topk<(E + 31) / 32>(lg, E, K, lane, my_idx, my_logit, pf_gu, L.exgu_expert, a.ex_dn, L.exdn_expert,
                                   dn0, dn1);
        if (rtid == 0) stamp(a, 4);
        if (lane < K) {
          ctl->act_e[lane] = (uint16_t)my_idx;
          ctl->act_mask[lane] = 1u;
          ctl->act_pb[lane] = (uint16_t)lane;
          ctl->pair_tok[lane] = 0;
          ctl->tok_pair[0][lane] = (uint8_t)lane;
          ctl->ids[0][lane] = my_idx;
        }
        if (lane == 0) {
          ctl->act_pb[K] = (uint16_t)K;
          ctl->U = ctl->abort ? 0 : K;
        }
        __syncwarp();
        if (lane == 0) plan();
        // routing weights: needed only from the down projection on
        const float mx = __shfl_sync(FULL, my_logit, 0);
        const float ex = lane < K ? __expf(my_logit - mx) : 0.f;
        const float Z = warp_sum(ex);
        const float wv = __fdividef(ex, Z);
        if (lane < K) {
          ctl->pair_w[lane] = wv;
          ctl->wts[0][lane] = wv;
        }
        if (lane == 0) ctl->sg[0] = __frcp_rn(1.0f + __expf(-__ldcg(lg + E)));
        if (cta == 0 && a.rec_ids) {
          int rank = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int oi = __shfl_sync(FULL, my_idx, i);
            rank += (i < K && oi < my_idx) ? 1 : 0;
          }
          if (lane < K) {
            a.rec_ids[rank] = my_idx;
            a.rec_w[rank] = wv;
          }
          if (lane == 0) a.rec_sg[0] = ctl->sg[0];
        }
      } else {
        if (!ctl->abort) {
#pragma unroll 1
          for (int t = rt; t < T; t += RW) {
            const float* lg = a.logits + (size_t)t * (E + 1);
            int my_idx;
            float my_logit;
            warp_topk<(E + 31) / 32>(lg, E, K, lane, my_idx, my_logit, pf_gu, L.exgu_expert, a.ex_dn,
                                     L.exdn_expert, dn0, dn1);
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
    if (!ctl->abort)
#pragma unroll 1
      for (int i = ctid; i < T * (Is / 16); i += CT) {
        const float4* src = reinterpret_cast<const float4*>(hst + (size_t)i * 16);
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
                  const float4* hv = reinterpret_cast<const float4*>(hst + (size_t)(tc + tt) * Is + cc * 16);
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
              for (int tt = 0; tt < nt; ++tt) shs[(tc + tt) * nrow + (r + rr - r0)] = rs[tt];
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
        if (!ctl->abort) {
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
      if (ONE) {
        // One token, U = K experts with one pair each, all their down items in the ring. Thread 0, which has
        // just seen every CTA's h, copies all U h vectors (already in the dot's lane order) into shared memory
        // with one bulk copy. A warp then takes one (expert, half of the CTA's rows): h into registers once,
        // rows four at a time as independent chains, and one transposed reduction per four rows.
        constexpr int NCL = (NC + 31) / 32;      // 16-column chunks per lane
        const int half = (nrow + 1) / 2;
        if (ctid == 0) {
          if (!ctl->abort && U > 0) {
            fence_proxy_async_global();
            mbar_expect_tx(&ctl->hbar, (uint32_t)(U * I * 4));
            bulk_g2s(hst, a.hbuf, (uint32_t)(U * I * 4), &ctl->hbar);
          } else {
            mbar_arrive(&ctl->hbar);
          }
        }
        if (!ctl->abort && !mbar_wait(&ctl->hbar, 0, a.timeout_ns)) set_error(a, ctl, ERR_WAIT_FULL);
        wstamp(a, cw, 2);
#pragma unroll 1
        for (int wi = cw; wi < 2 * U; wi += NCW) {
          const int aa = wi >> 1, rlo = (wi & 1) ? half : 0, rhi = (wi & 1) ? nrow : half;
          float4 hv[NCL][4];
          float hsum[NCL];
#pragma unroll
          for (int m = 0; m < NCL; ++m) {
            const int c = lane + 32 * m;
            hsum[m] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              hv[m][j] = (NC % 32 == 0 || c < NC) ? hst4[(size_t)aa * 4 * NC + j * NC + c] : make_float4(0.f, 0.f, 0.f, 0.f);
              hsum[m] += (hv[m][j].x + hv[m][j].y) + (hv[m][j].z + hv[m][j].w);
            }
          }
          // The expert's rows of this CTA are one ring item (the plan guarantees it for one token). A warp takes
          // eight consecutive rows from rlo: rows past rhi are read (they lie inside the same stage) and
          // dropped, so the eight dot products run unpredicated as independent chains.
          const uint8_t* item0 = stage_at(aa);
          float v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[q] = 0.f;
            const uint8_t* row = item0 + (rlo + q) * (int)L.DR;
#pragma unroll
            for (int m = 0; m < NCL; ++m) {
              const int c = lane + 32 * m;
              if (NC % 32 == 0 || c < NC) {
                const uint2 w = *reinterpret_cast<const uint2*>(row + c * 8);
                float2 qq[8];
                unpack_int4_quad(w.x & 0xFFFFu, qq[0], qq[1]);
                unpack_int4_quad(w.x >> 16, qq[2], qq[3]);
                unpack_int4_quad(w.y & 0xFFFFu, qq[4], qq[5]);
                unpack_int4_quad(w.y >> 16, qq[6], qq[7]);
                const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + I / 2 + (c >> 2) * 4));
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  acc = __ffma2_rn(qq[2 * j], make_float2(hv[m][j].x, hv[m][j].y), acc);
                  acc = __ffma2_rn(qq[2 * j + 1], make_float2(hv[m][j].z, hv[m][j].w), acc);
                }
                v[q] += sb.x * (acc.x + acc.y) + sb.y * hsum[m];
              }
            }
          }
          // transposed reduction of the eight values over the warp (9 shuffles): bit 4 of the lane keeps rows
          // 0-3 or 4-7, bit 3 one pair of those, bit 2 one row; then a butterfly over the last two bits.
          // Lane 4i ends with the sum for row rlo + i.
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
          if ((lane & 3) == 0 && rlo + idx < rhi) yv[(size_t)aa * nrow + rlo + idx] = z;
        }
        wstamp(a, cw, 3);
#pragma unroll 1
        for (int i = 0; i < U * dn_items; ++i) release();
      }
      if (!ONE) {
        // More tokens: every warp walks the active experts' down items in ring order. An expert's work is cut
        // into units of (half of this CTA's rows) x (up to PC of its token pairs), dealt round-robin to the
        // warps; a unit brings its pairs' h (lane-ordered rows of I floats) from L2 into registers and runs
        // eight rows as independent dot chains, one transposed reduction per pair.
        constexpr int PC = 2;
        constexpr int NCL = (NC + 31) / 32;
        const int half = (nrow + 1) / 2;
        int ui = 0;
#pragma unroll 1
        for (int aa = 0; aa < U; ++aa) {
          const int pb = ctl->act_pb[aa], na = (int)ctl->act_pb[aa + 1] - pb;
          const int nunits = 2 * ((na + PC - 1) / PC);
          const uint8_t* item = acquire();
#pragma unroll 1
          for (int k = 0; k < nunits; ++k, ++ui) {
            if (ui % NCW != cw || ctl->abort) continue;
            const int rlo = (k & 1) ? half : 0, rhi = (k & 1) ? nrow : half;
            const int p0 = pb + (k >> 1) * PC, np = min(PC, pb + na - p0);
            float4 hv[PC][NCL][4];
            float hsum[PC][NCL];
#pragma unroll
            for (int pp = 0; pp < PC; ++pp)
#pragma unroll
              for (int m = 0; m < NCL; ++m) {
                const int c = lane + 32 * m;
                hsum[pp][m] = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  hv[pp][m][j] = (pp < np && (NC % 32 == 0 || c < NC))
                                     ? __ldcg(reinterpret_cast<const float4*>(a.hbuf + (size_t)(p0 + pp) * I) + j * NC + c)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                  hsum[pp][m] += (hv[pp][m][j].x + hv[pp][m][j].y) + (hv[pp][m][j].z + hv[pp][m][j].w);
                }
              }
            float v[PC][8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
#pragma unroll
              for (int pp = 0; pp < PC; ++pp) v[pp][q] = 0.f;
              const uint8_t* row = item + (rlo + q) * (int)L.DR;
#pragma unroll
              for (int m = 0; m < NCL; ++m) {
                const int c = lane + 32 * m;
                if (NC % 32 == 0 || c < NC) {
                  const uint2 w = *reinterpret_cast<const uint2*>(row + c * 8);
                  float2 qq[8];
                  unpack_int4_quad(w.x & 0xFFFFu, qq[0], qq[1]);
                  unpack_int4_quad(w.x >> 16, qq[2], qq[3]);
                  unpack_int4_quad(w.y & 0xFFFFu, qq[4], qq[5]);
                  unpack_int4_quad(w.y >> 16, qq[6], qq[7]);
                  const float2 sb = h2f(*reinterpret_cast<const uint32_t*>(row + I / 2 + (c >> 2) * 4));
#pragma unroll
                  for (int pp = 0; pp < PC; ++pp) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      acc = __ffma2_rn(qq[2 * j], make_float2(hv[pp][m][j].x, hv[pp][m][j].y), acc);
                      acc = __ffma2_rn(qq[2 * j + 1], make_float2(hv[pp][m][j].z, hv[pp][m][j].w), acc);
                    }
                    v[pp][q] += sb.x * (acc.x + acc.y) + sb.y * hsum[pp][m];
                  }
                }
              }
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
          release();
        }
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
        if (a.gamma) v += __half2float(__ushort_as_half(a.x[(size_t)t * H + r0 + rr]));
        a.out[(size_t)t * H + r0 + rr] = __half_as_ushort(__float2half_rn(v));
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
  pl.hp = T == 1 ? L.K : 0;   // h vectors staged in shared memory (one token only)
  const Smem m = smem_map(L, T, grid, pl.hp);
  // 8 gate/up units (4 unit pairs, 4 warps) a stage. Each bulk copy costs a few hundred nanoseconds of the
  // SM's copy issue whatever its size, so fewer, larger copies land the routed weights sooner. With one token
  // the ring then wraps, but only in the routed down rows, whose stages free up long before they are needed.
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
  // The grid-wide counters need every CTA resident at once: one CTA per SM (its shared memory admits no
  // second) and grid <= SM count guarantee it once the SMs are free. The launch is programmatic-dependent
  // rather than cooperative: a dependent grid can start only after every CTA of this one has run
  // launch_dependents, so it never holds an SM that a CTA of this grid still waits for.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, pl.NS, pl.SS, pl.hp);
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
