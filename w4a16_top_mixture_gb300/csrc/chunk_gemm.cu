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
//   warps 0, 14  producers of the even (warp 0) or odd (warp 14) K-tiles: a bulk copy of the K-tile's weight
//              block (codes + pairs), TMA tensor loads of the activation rows (128-byte swizzled K-major) and a
//              bulk copy of the rows' sums over the K-tile's 64 columns, all on the stage's "full" barrier
//   warp 1     the MMAs of every K-tile (A from tensor memory, B from shared memory), committed to the stage's
//              "empty" barrier; it also owns TMEM. One thread issues all of the CTA's MMAs and commits: with two
//              issuing threads (alternate K-tiles), about one forward in thirty at 512 tokens came out with a
//              job at the start of a CTA's work corrupted.
// The producer and MMA warps step through their loops as whole warps, so that every copy and MMA operand is
// warp-uniform, and one elected lane issues the copies or the MMAs: with the loop in one lane, each issue cost
// that lane several hundred cycles (the MMAs of a K-tile: ~530 traced cycles, now ~75).
//   warps 2-9  dequantise, two groups of four warps taking alternate K-tiles: thread = band row = TMEM lane,
//              codes -> exact fp16 integers stored straight into the slot's A columns of tensor memory
//   warps 10-13 fold (thread = TMEM lane = band row) and, after the job's last K-tile, the epilogue
// K-tile gk uses shared-memory stage gk % nsg and tensor-memory slot gk % nt (A operand, accumulator and side
// buffer); there are more stages than slots so that more weight copies are in flight. A slot's accumulator is
// as wide as the launch's widest job, and it has a low-half accumulator only in phase 3 (the down
// projections, whose B is split into hi + lo halves): 8 slots fit the 512 columns when no job is wider than 32
// rows, 5 (phase 3: 3) at 64. Handoffs:
//   full[s]    the copies landed                                     (producer -> dequantisation)
//   a_ready[t] A and the side buffer are written                     (dequantisation -> MMA)
//   empty[s]   the dequantisation has read the stage and the MMAs have completed: the stage is free and the
//              accumulator holds the K-tile                          (-> producer, fold)
//   d_free[t]  the fold has read the accumulator and the side buffer; since the fold saw empty[s], the MMAs
//              that read A are complete too                          (fold -> dequantisation)
// Keeping A out of shared memory leaves the shared-memory pipe to the copies, the code loads and B.
// Every wait is bounded; on a timeout the CTA records an error bit and every role leaves its loops.
#include <mutex>
#include <cuda_fp16.h>
#include <stdint.h>

#include "chunk.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace moe {

namespace {

enum : int { GK_ROUTER = 0, GK_SHGU = 1, GK_SHDN = 2, GK_EXGU = 3, GK_EXDN = 4 };

constexpr int GTH = 480;                // 15 warps
constexpr int NSG_MAX = 16;             // shared-memory stages (the count depends on the phase, see Geo)
constexpr int NT_MAX = 8;               // tensor-memory slots (the count depends on the widest tile, see Slots)
// The stages share one area. A stage is weight block | B hi (up to 64 rows x 128 B, swizzled) | [B lo], each
// part 1024-byte aligned (the 128-byte swizzle's period). Its size depends on the phase, and so does the number
// of stages: the fewer bytes a K-tile needs, the more K-tiles are in flight (the copies' latency is what the
// pipeline has to cover).
constexpr int ST_AREA = 186368;
struct Geo {
  int nsg, bytes, bhi, blo;
};
__host__ __device__ constexpr Geo geo_of(int phase) {
  return phase == 1 ? Geo{10, 17408, 9216, 9216}       // int8 router / shared gate-up blocks, B hi
         : phase == 2 ? Geo{14, 13312, 5120, 5120}     // int4 expert gate/up blocks, B hi
                      : Geo{7, 25600, 9216, 17408};    // int4 / int8 down blocks, B hi and lo
}
static_assert(geo_of(1).nsg * geo_of(1).bytes <= ST_AREA && geo_of(2).nsg * geo_of(2).bytes <= ST_AREA &&
                  geo_of(3).nsg * geo_of(3).bytes <= ST_AREA && geo_of(2).nsg <= NSG_MAX,
              "stages");
static_assert(GEMM_BLK8 <= 9216 && GEMM_BLK4 <= 5120, "weight block fits before B");
constexpr int ST_W = 0;
constexpr int S_SIDE = ST_AREA;                     // NT_MAX side buffers: (s, b) of 128 rows, 64 row sums
constexpr int SIDE_BYTES = 128 * 4 + 64 * 4;
constexpr int S_SUMS = S_SIDE + NT_MAX * SIDE_BYTES;  // per stage: the K-tile's run of activation sums
constexpr int SUMS_BYTES = SUM_RUN * 4;
static_assert(SUMS_BYTES % 16 == 0 && S_SUMS % 16 == 0, "bulk-copy alignment");
constexpr int S_EP = S_SUMS + NSG_MAX * SUMS_BYTES;  // epilogue staging of a job's accumulator: [128][65]
constexpr int S_BAR = S_EP + 128 * 65 * 4;
constexpr int S_BYTES = S_BAR + 512;
constexpr int GEMM_SMEM = S_BYTES + 1024;           // + alignment slack
static_assert(GEMM_SMEM <= 232448, "shared memory");
constexpr uint32_t ERR_GEMM_WAIT = 512u;

struct Job {
  int kind, m, e;
  const uint8_t* w;       // weight block of K-tile 0 of the band
  int ktiles, int8;
  int bmap, lomap;        // tensor maps of the activations and of their low halves (-1: none)
  int row0, cnt, n;       // first activation row, rows, MMA N (cnt rounded up to 16)
  const float* sum;       // K-tile-major sums of the activation rows
  int sstride;            // their row stride
};

// a ring position (tensor-memory slot or shared-memory stage) of a role's current K-tile and the parity of the
// position's current use
struct SlotRing {
  int t = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int nt) {
    if (++t == nt) { t = 0; ph ^= 1u; }
  }
};

// Job j of the phase. Phases 2 and 3 take the expert row-tile count (ngroups) and job j's row-tile entry gr
// (S.groups[j % ngroups] for the expert jobs) from the caller, which loads them ahead of time.
// Token tiles (phase 1, and the shared down of phase 3) are tw rows wide.
__device__ __forceinline__ bool decode_job(const GemmArgs& g, int j, int ngroups, int tw, int4 gr, Job& jb) {
  const GemmLayout& G = g.G;
  const ChunkScratch& S = g.S;
  const int H = G.H, I = G.I, Is = G.Is, T = g.T;
  const int NTT = (T + tw - 1) / tw;
  jb.e = 0;
  jb.lomap = -1;
  auto token_tile = [&](int nt) {
    jb.row0 = nt * tw;
    jb.cnt = min(tw, T - jb.row0);
  };
  if (g.phase == 1) {
    const int MTr = G.Mr / 128, MTs = 2 * Is / 128;
    if (j < MTr * NTT) {
      jb.kind = GK_ROUTER; jb.m = j % MTr; token_tile(j / MTr);
      jb.w = G.gr + (size_t)jb.m * (H / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = H / 64;
      jb.bmap = CM_XP; jb.sum = S.sum_xp; jb.sstride = S.sp;
    } else {
      j -= MTr * NTT;
      if (j >= MTs * NTT) return false;
      jb.kind = GK_SHGU; jb.m = j % MTs; token_tile(j / MTs);
      jb.w = G.gsgu + (size_t)jb.m * (H / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = H / 64;
      jb.bmap = CM_XP; jb.sum = S.sum_xp; jb.sstride = S.sp;
    }
  } else {
    const int MTg = 2 * I / 128, MTd = H / 128;
    const int nex = (g.phase == 2 ? MTg : MTd) * ngroups;   // expert jobs; phase 3 then the shared down
    if (j < nex) {
      // band-major: the row tiles of one expert for one band are consecutive jobs (they share the band's
      // weights through L2)
      const int m = j / ngroups;
      jb.m = m; jb.e = gr.x; jb.row0 = gr.y; jb.cnt = gr.z; jb.int8 = 0;
      if (g.phase == 2) {
        jb.kind = GK_EXGU;
        jb.w = G.gegu + (size_t)gr.x * G.gegu_expert + (size_t)m * (H / 64) * GEMM_BLK4; jb.ktiles = H / 64;
        jb.bmap = CM_XS; jb.sum = S.sum_xs; jb.sstride = S.sr;
      } else {
        jb.kind = GK_EXDN;
        jb.w = G.gedn + (size_t)gr.x * G.gedn_expert + (size_t)m * (I / 64) * GEMM_BLK4; jb.ktiles = I / 64;
        jb.bmap = CM_HH; jb.lomap = CM_HHLO; jb.sum = S.sum_hh; jb.sstride = S.sr;
      }
    } else {
      j -= nex;
      if (g.phase != 3 || j >= MTd * NTT) return false;
      jb.kind = GK_SHDN; jb.m = j % MTd; token_tile(j / MTd);
      jb.w = G.gsdn + (size_t)jb.m * (Is / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = Is / 64;
      jb.bmap = CM_HS; jb.lomap = CM_HSLO; jb.sum = S.sum_hs; jb.sstride = S.sp;
    }
  }
  jb.n = (jb.cnt + 15) & ~15;
  return jb.cnt > 0;
}

// A role's walk over its CTA's jobs j = blockIdx.x + k * gridDim.x. The row-tile entry of the next job is
// loaded while the current one runs, so a job change costs no global-memory round trip.
struct JobIter {
  int j, ngroups, tw;
  int4 gr;
};
__device__ __forceinline__ int4 job_group(const GemmArgs& g, int ngroups, int j) {
  const int MT = g.phase == 2 ? 2 * g.G.I / 128 : g.G.H / 128;
  if (g.phase == 1 || ngroups <= 0 || j >= MT * ngroups) return make_int4(0, 0, 0, 0);
  return g.S.groups[j % ngroups];
}
__device__ __forceinline__ void job_begin(const GemmArgs& g, int ngroups, int tw, JobIter& it) {
  it.j = blockIdx.x;
  it.ngroups = ngroups;
  it.tw = tw;
  it.gr = job_group(g, it.ngroups, it.j);
}
__device__ __forceinline__ bool job_next(const GemmArgs& g, JobIter& it, Job& jb) {
  const bool ok = decode_job(g, it.j, it.ngroups, it.tw, it.gr, jb);
  it.j += gridDim.x;
  it.gr = job_group(g, it.ngroups, it.j);
  return ok;
}

struct Bars {
  uint64_t full[NSG_MAX], empty[NSG_MAX], a_ready[NT_MAX], d_free[NT_MAX];
  uint64_t acc_full[2], acc_free[2];   // a job's accumulator (job parity) is complete / has been read
  uint64_t fold_sync;   // the four fold warps meet here in the SwiGLU epilogue (a bounded wait)
  uint32_t tslot;
  int ngroups, tw;      // the launch's row-tile count and token-tile width, read once
  volatile int abort;
};
static_assert(sizeof(Bars) <= S_BYTES - S_BAR, "barrier area");

// debug stamps (CTA 0, first 64 K-tiles): events 0 producer issued, 1 dequant saw the stage, 2 dequant done,
// 3 MMA issued, 4 fold saw the accumulator, 5 fold done, 6 MMA saw A ready
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
  // bounded wait on phase parity `ph` of `b`; false (and the CTA aborts) on a timeout; a wait that does not
  // complete at once gives up straight away if the CTA has already aborted
  auto wait = [&](uint64_t* b, uint32_t ph) -> bool {
    if (mbar_try_wait(b, ph)) return true;
    if (bar->abort) return false;
    if (!mbar_wait_slow(b, ph, to)) { fail(); return false; }
    return true;
  };

  if (tid == 0) {
    for (int s = 0; s < NSG_MAX; ++s) {
      mbar_init(&bar->full[s], 1);          // the producer's expect-tx arrival
      mbar_init(&bar->empty[s], 4 + 1);     // dequant warps (codes, pairs, sums read) + MMA commit (B read)
    }
    for (int i = 0; i < NT_MAX; ++i) {
      mbar_init(&bar->a_ready[i], 4);
      mbar_init(&bar->d_free[i], 4);
    }
    mbar_init(&bar->fold_sync, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar->acc_full[b], 1);   // the MMA issuer's commit after the job's last K-tile
      mbar_init(&bar->acc_free[b], 4);   // the fold warps, once they have read the accumulator
    }
    bar->abort = 0;
    // phase 1 tiles the tokens 64 at a time; phases 2 and 3 take the bucketing's row tiles, and phase 3 tiles
    // the shared down's tokens as wide as the widest row tile, so no job is wider than that
    bar->ngroups = g.phase == 1 ? 0 : g.S.ctl[0];
    bar->tw = g.phase == 1 ? CHUNK_NT : min(CHUNK_NT, max(16, (g.S.ctl[1] + 15) & ~15));
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(&bar->tslot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tslot;
  const Geo geo = geo_of(g.phase);
  const uint32_t NSG = (uint32_t)geo.nsg;
  const int ngroups = bar->ngroups, tw = bar->tw;
  // tensor memory: two job accumulators (job parity), each aw columns (aw = the widest job's N rounded up to
  // 32) plus, in phase 3, a low-half accumulator of aw more; then the A slots, 64 columns each: A1 = fp16(s q)
  // and A2 = s q - A1 (exact), 128 rows x 64 K each
  const bool lo_phase = g.phase == 3;
  const uint32_t aw = (uint32_t)((min(tw, g.phase == 1 ? ((min(g.T, CHUNK_NT) + 15) & ~15) : CHUNK_NT) + 31) & ~31);
  const uint32_t dcols = lo_phase ? 2 * aw : aw, tlo = aw, a0 = 2 * dcols;
  const int nt = min(NT_MAX, (int)((512 - a0) / 64));
  float* sums = reinterpret_cast<float*>(smem + S_SUMS);   // [NSG_MAX][SUM_RUN]

  if (warp == 0 || warp == 14) {
    // ------------------------------------------------------------------ producers
    // Warp 0 fills the stages of the even K-tiles, warp 14 those of the odd ones. The whole warp steps through
    // the loop, so every copy operand is warp-uniform, and one elected lane arms the stage and issues its
    // copies: the weight block and the sums run (1-D bulk copies), then B hi and B lo (tensor loads).
    const uint32_t par = warp == 0 ? 0u : 1u;
    uint32_t gk = 0;
    bool run = true;
    // test hook: CTA 0 never arms or fills the stage of its first K-tile, so the roles waiting for it time
    // out and the CTA aborts
    const bool withhold = g.skip && blockIdx.x == 0;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sr;
    while (run && job_next(g, it, jb)) {
      const int blk = jb.int8 ? GEMM_BLK8 : GEMM_BLK4;
      const int box = jb.n <= 16 ? 0 : jb.n <= 32 ? 1 : 2;
      const bool lo = jb.lomap >= 0;
      const uint32_t tx = (uint32_t)(blk + SUMS_BYTES) + (16u << box) * 128u * (lo ? 2u : 1u);
      // the K-tile's sums for the tile's rows: SUM_RUN floats from the first row rounded down to a multiple of
      // 4 (16-byte aligned, the row strides being multiples of 4 floats)
      const float* srun = jb.sum + (jb.row0 & ~3);
      const CUtensorMap* mhi = &g.maps.m[jb.bmap][box];
      const CUtensorMap* mlo = &g.maps.m[lo ? jb.lomap : jb.bmap][box];
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk, sr.next(NSG)) {
        if ((gk & 1u) != par) continue;
        const int s = sr.t;
        const bool ok = gk < NSG || wait(&bar->empty[s], sr.ph ^ 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) { run = false; break; }
        if (withhold && gk == 0) continue;
        uint8_t* st = smem + s * geo.bytes;
        if (elect_one()) {
          mbar_expect_tx(&bar->full[s], tx);
          bulk_g2s(st + ST_W, jb.w + (size_t)kt * blk, (uint32_t)blk, &bar->full[s]);
          bulk_g2s(sums + s * SUM_RUN, srun + (size_t)kt * jb.sstride, (uint32_t)SUMS_BYTES, &bar->full[s]);
          tma_load_2d(st + geo.bhi, mhi, kt * 64, jb.row0, &bar->full[s]);
          if (lo) tma_load_2d(st + geo.blo, mlo, kt * 64, jb.row0, &bar->full[s]);
          GSTAMP(0, gk);
        }
        __syncwarp();
      }
    }
    // drain: every copy this warp issued must have landed before the CTA leaves (the withheld one was never
    // issued); only the last NSG K-tiles can still be in flight
    if (lane == 0) {
      const uint32_t cnt = gk < (uint32_t)NSG ? gk : (uint32_t)NSG;
      for (uint32_t q = gk - cnt; q < gk; ++q)
        if ((q & 1u) == par && !(withhold && q == 0)) mbar_wait(&bar->full[q % NSG], (q / NSG) & 1u, to);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    // The whole warp steps through the loop and waits, so the descriptors and TMEM addresses are warp-uniform;
    // one elected lane (the same one every time) issues the MMAs and the commit.
    uint32_t gk = 0, njob = 0;
    bool run = true;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sl, sr;
    while (run && job_next(g, it, jb)) {
      const uint32_t idesc = umma_idesc_f16(128, jb.n);
      const bool lo = jb.lomap >= 0;
      const uint32_t b = njob & 1u, d = tmem + b * dcols;
      // the job accumulates in accumulator b, which the fold of job njob - 2 must have read
      {
        const bool ok = njob < 2 || wait(&bar->acc_free[b], ((njob >> 1) - 1) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) { run = false; break; }
      }
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk, sl.next(nt), sr.next(NSG)) {
        const int s = sr.t, t = sl.t;
        // a_ready implies full[s] and that the fold of K-tile gk - nt released slot t (the dequantisation
        // waited for both)
        const bool ok = wait(&bar->a_ready[t], sl.ph);
        if (!__all_sync(0xFFFFFFFFu, ok)) { run = false; break; }
        tc_fence_after();
        // B descriptors of the stage; a K step of 16 elements advances the start address by 32 bytes (2 units)
        const uint8_t* st = smem + s * geo.bytes;
        const uint64_t bh = umma_desc_sw128(smem_u32(st + geo.bhi)), bl = umma_desc_sw128(smem_u32(st + geo.blo));
        const uint32_t a = tmem + a0 + 64u * (uint32_t)t;
        if (elect_one()) {
          GSTAMP(6, gk);
          // D += A1 B + A2 B: the exact products s q x, summed over the whole job
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            umma_f16_ts(d, a + 8 * ks, bh + 2 * ks, idesc, (kt > 0 || ks > 0) ? 1u : 0u);
            umma_f16_ts(d, a + 32 + 8 * ks, bh + 2 * ks, idesc, 1u);
          }
          // the low halves of the activations: A2's share there is below fp32 resolution of the sum
          if (lo)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f16_ts(d + tlo, a + 8 * ks, bl + 2 * ks, idesc, (kt > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bar->empty[s]);
          if (kt == jb.ktiles - 1) umma_commit(&bar->acc_full[b]);
          GSTAMP(3, gk);
        }
        __syncwarp();
      }
      ++njob;
    }
    // the last MMAs must have completed before TMEM is released (a commit tracks all earlier MMAs of its thread)
    if (lane == 0 && gk > 0) mbar_wait(&bar->empty[(gk - 1) % NSG], ((gk - 1) / NSG) & 1u, to);
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------------------------------------ dequantise
    const int grp = (warp - 2) >> 2;          // this group takes the K-tiles gk with gk % 2 == grp
    const int r = (warp & 3) * 32 + lane;     // band row = the TMEM lane this warp may access
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const __half2 k1024 = __float2half2_rn(1024.0f), k16 = __float2half2_rn(0.0625f), k64 = __float2half2_rn(-64.0f);
    uint32_t gk = 0;
    bool run = true;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sl, sr;
    while (run && job_next(g, it, jb)) {
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk, sl.next(nt), sr.next(NSG)) {
        if ((int)(gk & 1u) != grp) continue;
        const int s = sr.t, t = sl.t;
        // d_free[t] of K-tile gk - nt: the fold is done with slot t, and the MMAs that read its A are complete
        if (!wait(&bar->full[s], sr.ph) ||
            (gk >= (uint32_t)nt && !wait(&bar->d_free[t], sl.ph ^ 1u))) {
          run = false;
          break;
        }
        if (r == 0) GSTAMP(1, gk);
        const uint8_t* st = smem + s * geo.bytes + ST_W;
        // the fold's share of the stage goes to the side buffer, so the stage is free once the MMA has read B:
        // row r's (s, b) pair and the sums of the tile's activation rows
        {
          uint32_t* side = reinterpret_cast<uint32_t*>(smem + S_SIDE + t * SIDE_BYTES);
          side[r] = *reinterpret_cast<const uint32_t*>(st + 128 * (jb.int8 ? 64 : 32) + r * 4);   // (s, b)
          if (r < CHUNK_NT) reinterpret_cast<float*>(side)[128 + r] = sums[s * SUM_RUN + (jb.row0 & 3) + r];
        }
        // row r of A1 and A2 in K order: column 4c + k holds the pair k of 8-column block c, A1 = fp16(s q),
        // A2 = s q - A1 (exact: s q is a multiple of s's unit in the last place with at most 19 significant bits,
        // so the rounding residual has at most 9 and is a multiple of that unit, never below 2^-24). Two halves of
        // 16 columns each, stored as soon as they are made.
        const uint32_t sbw = *reinterpret_cast<const uint32_t*>(st + 128 * (jb.int8 ? 64 : 32) + r * 4);
        const __half2 s2 = __low2half2(*reinterpret_cast<const __half2*>(&sbw));
        const uint32_t ta = trow + a0 + 64u * (uint32_t)t;
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          uint32_t a1[16], a2[16];
          auto put = [&](int i, __half2 q) {
            const __half2 h1 = __hmul2(q, s2);
            const __half2 h2 = __hfma2(q, s2, __hneg2(h1));
            a1[i] = *reinterpret_cast<const uint32_t*>(&h1);
            a2[i] = *reinterpret_cast<const uint32_t*>(&h2);
          };
          if (jb.int8) {
            const uint8_t* codes = st + r * 64 + hlf * 32;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint2 w = *reinterpret_cast<const uint2*>(codes + c * 8);
              uint32_t v[4];
              int8_block_pairs(w.x, w.y, v);
#pragma unroll
              for (int k = 0; k < 4; ++k) put(4 * c + k, __hsub2(*reinterpret_cast<const __half2*>(&v[k]), k1024));
            }
          } else {
            const uint4 w4 = *reinterpret_cast<const uint4*>(st + r * 32 + hlf * 16);
            const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[4];
              int4_word_pairs(wd[c], v);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const __half2 h = *reinterpret_cast<const __half2*>(&v[k]);
                // exact codes: 1024 + q -> q; 1024 + 16 q (odd pairs) -> q
                put(4 * c + k, (k & 1) ? __hfma2(h, k16, k64) : __hsub2(h, k1024));
              }
            }
          }
          tmem_st16(ta + 16u * hlf, a1);
          tmem_st16(ta + 32u + 16u * hlf, a2);
        }
        tmem_wait_st();
        tc_fence_before();   // the MMAs read A after the a_ready handoff
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar->a_ready[t]);
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
    float* ep = reinterpret_cast<float*>(smem + S_EP);      // [128 rows][65] the job's accumulator
    const GemmLayout& G = g.G;
    const ChunkScratch& S = g.S;
    uint32_t fph = 0, njob = 0;
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
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sl, sr;
    while (run && job_next(g, it, jb)) {
      float acc[CHUNK_NT];
#pragma unroll
      for (int i = 0; i < CHUNK_NT; ++i) acc[i] = 0.f;
      for (int kt = 0; kt < jb.ktiles; ++kt, ++gk, sl.next(nt), sr.next(NSG)) {
        const int s = sr.t, t = sl.t;
        // empty[s] completes once the MMAs have finished and the dequantisation (which wrote the side buffer
        // before arriving) is done
        if (!wait(&bar->empty[s], sr.ph)) {
          run = false;
          break;
        }
        tc_fence_after();
        if (r == 0) GSTAMP(4, gk);
        const uint32_t* side = reinterpret_cast<const uint32_t*>(smem + S_SIDE + t * SIDE_BYTES);
        const float2 sb = h2f(side[r]);
        const float4* xs4 = reinterpret_cast<const float4*>(side + 128);
        // the affine's offset part of the group: acc += b * sum(x) (the scaled codes accumulate in TMEM)
#pragma unroll
        for (int c0 = 0; c0 < CHUNK_NT; c0 += 16) {
          if (c0 < jb.n) {
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 x4 = xs4[(c0 + i) >> 2];
              acc[c0 + i] = fmaf(sb.y, x4.x, acc[c0 + i]);
              acc[c0 + i + 1] = fmaf(sb.y, x4.y, acc[c0 + i + 1]);
              acc[c0 + i + 2] = fmaf(sb.y, x4.z, acc[c0 + i + 2]);
              acc[c0 + i + 3] = fmaf(sb.y, x4.w, acc[c0 + i + 3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->d_free[t]);
        if (r == 0) GSTAMP(5, gk);
      }
      if (!run) break;
      // ---- the job's accumulator: s * sum(q x) over all its K-tiles (+ the low halves' share / 4096)
      {
        const uint32_t b = njob & 1u;
        if (!wait(&bar->acc_full[b], (njob >> 1) & 1u)) break;
        tc_fence_after();
        const uint32_t d = trow + b * dcols;
#pragma unroll
        for (int c0 = 0; c0 < CHUNK_NT; c0 += 16) {
          if (c0 < jb.n) {
            uint32_t v[16];
            tmem_ld16_nowait(d + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[c0 + i] += __uint_as_float(v[i]);
            if (jb.lomap >= 0) {
              tmem_ld16_nowait(d + tlo + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[c0 + i] = fmaf(__uint_as_float(v[i]), 1.0f / 4096.0f, acc[c0 + i]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->acc_free[b]);
        ++njob;
      }
      // ---- epilogue. The accumulator goes to shared memory (its register indices are compile-time, so this
      // is the only unrolled step), then short loops over the tile's tokens write the results: the code that
      // runs once per job stays small.
#pragma unroll
      for (int c0 = 0; c0 < CHUNK_NT; c0 += 16)
        if (c0 < jb.n)
#pragma unroll
          for (int i = 0; i < 16; ++i) ep[r * 65 + c0 + i] = acc[c0 + i];
      if (!fold_sync()) break;
      const int cnt = jb.cnt;
      if (jb.kind == GK_ROUTER) {
        // thread = band row (router output row), tokens in a loop; consecutive rows on consecutive lanes
        const int er = jb.m * 128 + r;
        if (er <= G.E)
#pragma unroll 4
          for (int i = 0; i < cnt; ++i) S.logits[(size_t)(jb.row0 + i) * (G.E + 1) + er] = ep[r * 65 + i];
      } else if (jb.kind == GK_SHDN || jb.kind == GK_EXDN) {
        float* dst = jb.kind == GK_SHDN ? S.ys : S.y;
#pragma unroll 4
        for (int i = 0; i < cnt; ++i) dst[(size_t)(jb.row0 + i) * G.H + jb.m * 128 + r] = ep[r * 65 + i];
      } else {
        // SwiGLU: rows 0-63 are gate units 64m.., rows 64-127 the matching up units. h = silu(g) * u is split
        // into fp16 hi + lo/4096 halves, the down projection's B operand; the 64 units are group m of the down
        // projection's reduction, so the group's sum (of hi + lo/4096, the values the MMAs see) is made here
        // too. Warp = token (4 at a time), lane = units u and u + 32.
        const bool sh = jb.kind == GK_SHGU;
        const int kd = sh ? G.Is : G.I;
        uint16_t* dhi = sh ? S.hs : S.hh;
        uint16_t* dlo = sh ? S.hs_lo : S.hh_lo;
        float* dsum = (sh ? S.sum_hs : S.sum_hh) + (size_t)jb.m * (sh ? S.sp : S.sr);
        const int pos0 = p8u(jb.m * 64 + lane), pos1 = p8u(jb.m * 64 + 32 + lane);
#pragma unroll 1
        for (int i = q4; i < cnt; i += 4) {
          float part = 0.f;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int u = lane + 32 * hf;
            const float h = silu_c(ep[u * 65 + i]) * ep[(u + 64) * 65 + i];
            const __half hh = __float2half_rn(h);
            const __half hl = __float2half_rn((h - __half2float(hh)) * 4096.0f);
            const size_t o = (size_t)(jb.row0 + i) * kd + (hf ? pos1 : pos0);
            dhi[o] = __half_as_ushort(hh);
            dlo[o] = __half_as_ushort(hl);
            part += fmaf(__half2float(hl), 1.0f / 4096.0f, __half2float(hh));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
          if (lane == 0) dsum[jb.row0 + i] = part;
        }
      }
      if (!fold_sync()) break;   // the staging buffer is free for the next job
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

static std::mutex g_gemm_attr_mutex;

cudaError_t chunk_gemm_launch(const GemmArgs& g, int grid, cudaStream_t st) {
  // the shared-memory limit is a per-device setting of the function: raise it once on every device used
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_gemm_attr_mutex);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(k_chunk_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  k_chunk_gemm<<<grid, GTH, GEMM_SMEM, st>>>(g);
  return cudaGetLastError();
}

}  // namespace moe
