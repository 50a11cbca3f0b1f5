// Grouped GEMMs of the prompt-chunk path on the tcgen05 tensor cores.
//
// A job is one 128-row band of a weight matrix (an expert's gate/up or down, the router, the shared expert)
// against one tile of up to 64 activation rows (tokens). A weight is w = s q + b per group of 64 inputs
// (K-tile). For every K-tile the dequantisation writes A1 = fp16(s q) and A2 = s q - A1 into tensor memory:
// the residual is exact (s q is a multiple of s's unit in the last place with at most 19 significant bits), so
// A1 + A2 = s q exactly, and the MMAs add A1 x + A2 x into one fp32 accumulator for the whole job. The offset
// term sum_g b_g sum(x over group g) is one more MMA per job: its A holds each K-tile's b (exact in fp16, the
// dequantisation writes one column per K-tile), its B the activation rows' group sums as fp16 hi + lo (one
// 128-byte row per activation row, made by the kernel that writes the row). The B operand of the down
// projections is h split into fp16 hi + lo/4096 halves; the low halves multiply A1 into a second accumulator
// (A2's share there is below the fp32 resolution of the sum).
//
// Persistent CTAs (one per SM, 20 warps) take jobs j = blockIdx.x + k * gridDim.x. Warp roles, all stepping
// through the same jobs and K-tiles and handing stages over on mbarriers:
//   warps 0, 18, 19  producers, each of every third K-tile: a bulk copy of the K-tile's weight block (codes +
//              pairs) and TMA tensor loads of the activation rows (128-byte swizzled K-major), on the stage's
//              "full" barrier; the producer of a job's first K-tile also loads the job's group-sum rows into
//              the job's bias tile
//   warp 1     the MMAs (A from tensor memory, B from shared memory) and their commits; it also owns TMEM. One
//              thread issues all of the CTA's MMAs and commits: with two issuing threads (alternate K-tiles),
//              about one forward in thirty at 512 tokens came out with a job at the start of a CTA's work
//              corrupted.
//   warps 2-13 dequantise, three groups of four warps, each taking every third K-tile: thread = band row =
//              TMEM lane
//   warps 14-17 the epilogue of each job (thread = TMEM lane = band row)
// The producer and MMA warps step through their loops as whole warps, so that every copy and MMA operand is
// warp-uniform, and one elected lane issues the copies or the MMAs: with the loop in one lane, each issue cost
// that lane several hundred cycles (the MMAs of a K-tile: ~530 traced cycles, now ~75).
//
// Tensor memory: two job accumulators (job parity; the epilogue of one job overlaps the next), each as wide as
// the launch's widest job plus, in phase 3, as much again for the low half; two bias A operands of 32 columns
// (job parity); then the A slots of 64 columns (A1 | A2). K-tile gk uses stage gk % nsg and A slot gk % nt.
// Handoffs:
//   full[s]        the copies landed                                          (producer -> dequantisation)
//   a_ready[t]     A slot t and the K-tile's bias column are written           (dequantisation -> MMA)
//   empty[s]       the dequantisation has read the stage and the MMAs have completed (-> producer)
//   a_free[t]      the MMAs that read A slot t completed                      (MMA commit -> dequantisation)
//   bb_full[p]     the bias tile of a job of parity p landed                  (producer -> MMA)
//   acc_full[p]    a job's MMAs, its bias MMA included, completed: the accumulator, the bias tile and the
//                  bias A of parity p are final and read                      (MMA commit -> epilogue, producer,
//                                                                              dequantisation)
//   acc_free[p]    the epilogue has read the accumulator of parity p          (epilogue -> MMA)
// A wait on a phase parity passes at once if the barrier is still one phase behind (its previous phase has the
// other parity), so no role may wait for a barrier's use u + 1 while its use u can still be pending. The three
// dequantisation groups step through the stages independently, so a group first waits for a stage's previous
// release (empty) before its fill (full). Every other barrier is waited on in the order of its uses.
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

constexpr int NDQ = 3;                  // dequantisation groups
constexpr int NPR = 3;                  // producer warps
constexpr int GTH = 640;                // 20 warps
constexpr int WEP = 2 + 4 * NDQ;        // first epilogue warp
constexpr int NSG_MAX = 16;             // shared-memory stages (the count depends on the phase, see Geo)
constexpr int NT_MAX = 8;               // A slots in tensor memory (the count depends on the widest job)
// The stages share one area. A stage is weight block | B hi (up to 64 rows x 128 B, swizzled) | [B lo], each
// part 1024-byte aligned (the 128-byte swizzle's period). Its size depends on the phase, and so does the number
// of stages: the fewer bytes a K-tile needs, the more K-tiles are in flight (the copies' latency is what the
// pipeline has to cover).
constexpr int ST_AREA = 179200;
struct Geo {
  int nsg, bytes, bhi, blo;
};
__host__ __device__ constexpr Geo geo_of(int phase) {
  return phase != 3 ? Geo{10, 17408, 9216, 9216}       // int8 router; int4 expert / int8 shared gate/up; B hi
                    : Geo{7, 25600, 9216, 17408};      // int4 / int8 down blocks, B hi and lo
}
static_assert(geo_of(1).nsg * geo_of(1).bytes <= ST_AREA && geo_of(2).nsg * geo_of(2).bytes <= ST_AREA &&
                  geo_of(3).nsg * geo_of(3).bytes <= ST_AREA && geo_of(1).nsg <= NSG_MAX,
              "stages");
static_assert(GEMM_BLK8 <= 9216 && GEMM_BLK4 <= 5120, "weight block fits before B");
static_assert(GSUM_COLS * 2 == 128, "a group-sum row is one 128-byte swizzle row");
constexpr int ST_W = 0;
constexpr int S_BB = ST_AREA;                       // two bias tiles (job parity): 64 rows x 128 B, swizzled
constexpr int BB_BYTES = CHUNK_NT * 128;
constexpr int S_EP = S_BB + 2 * BB_BYTES;           // epilogue staging of a job's accumulator: [128][65]
constexpr int S_BAR = S_EP + 128 * 65 * 4;
constexpr int S_BYTES = S_BAR + 512;
constexpr int GEMM_SMEM = S_BYTES + 1024;           // + alignment slack
static_assert(S_BB % 1024 == 0 && BB_BYTES % 1024 == 0, "swizzled tiles are 1024-byte aligned");
static_assert(GEMM_SMEM <= 232448, "shared memory");
constexpr uint32_t ERR_GEMM_WAIT = 512u;

struct Job {
  int kind, m, e;
  const uint8_t* w;       // weight block of K-tile 0 of the band
  int ktiles, int8;
  int k0, part;           // the job's first K-tile and K part (the router's split; 0 otherwise)
  int bmap, lomap;        // tensor maps of the activations and of their low halves (-1: none)
  int row0, cnt, n;       // first activation row, rows, MMA N (cnt rounded up to 16)
  int gmap;               // tensor map of the activation rows' group sums
};

// a ring position (tensor-memory slot or shared-memory stage) of a role's current K-tile and the parity of the
// position's current use
struct SlotRing {
  int t = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int nt) {
    if (++t == nt) { t = 0; ph ^= 1u; }
  }
  // n steps at once, n <= nt
  __device__ __forceinline__ void adv(int n, int nt) {
    t += n;
    if (t >= nt) { t -= nt; ph ^= 1u; }
  }
};

// Job j of the phase. Phases 2 and 3 take the expert row-tile count (ngroups) and job j's row-tile entry gr
// (S.groups[j % ngroups] for the expert jobs) from the caller, which loads them ahead of time.
// Phase 1: the router bands by token tile (tw = CHUNK_NT rows) and K part. Phase 2: the expert gate/up jobs,
// then the shared gate/up bands by token tiles of CHUNK_NT. Phase 3: the expert down jobs, then the shared down
// bands by token tiles of tw rows.
__device__ __forceinline__ bool decode_job(const GemmArgs& g, int j, int ngroups, int tw, int4 gr, Job& jb) {
  const GemmLayout& G = g.G;
  const int H = G.H, I = G.I, Is = G.Is, T = g.T;
  const int NTT = (T + tw - 1) / tw;
  jb.e = 0;
  jb.lomap = -1;
  jb.k0 = 0;
  jb.part = 0;
  auto token_tile = [&](int nt) {
    jb.row0 = nt * tw;
    jb.cnt = min(tw, T - jb.row0);
  };
  if (g.phase == 1) {
    // the router bands, each token tile's K cut into router_parts parts (jobs of their own)
    const int MTr = G.Mr / 128, KT = H / 64, kpp = router_kpp(KT), NP = router_parts(KT);
    if (j >= MTr * NTT * NP) return false;
    const int rest = j / MTr;
    jb.kind = GK_ROUTER; jb.m = j % MTr; token_tile(rest % NTT);
    jb.part = rest / NTT; jb.k0 = jb.part * kpp; jb.ktiles = min(kpp, KT - jb.k0);
    jb.w = G.gr + (size_t)jb.m * KT * GEMM_BLK8; jb.int8 = 1;
    jb.bmap = CM_XP; jb.gmap = CM_GXP;
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
        jb.bmap = CM_XS; jb.gmap = CM_GXS;
      } else {
        jb.kind = GK_EXDN;
        jb.w = G.gedn + (size_t)gr.x * G.gedn_expert + (size_t)m * (I / 64) * GEMM_BLK4; jb.ktiles = I / 64;
        jb.bmap = CM_HH; jb.lomap = CM_HHLO; jb.gmap = CM_GHH;
      }
    } else if (g.phase == 2) {
      // then the shared expert's gate/up bands, in token tiles of CHUNK_NT
      j -= nex;
      const int MTs = 2 * Is / 128, NTS = (T + CHUNK_NT - 1) / CHUNK_NT;
      if (j >= MTs * NTS) return false;
      jb.kind = GK_SHGU; jb.m = j % MTs;
      jb.row0 = (j / MTs) * CHUNK_NT;
      jb.cnt = min(CHUNK_NT, T - jb.row0);
      jb.w = G.gsgu + (size_t)jb.m * (H / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = H / 64;
      jb.bmap = CM_XP; jb.gmap = CM_GXP;
    } else {
      j -= nex;
      if (j >= MTd * NTT) return false;
      jb.kind = GK_SHDN; jb.m = j % MTd; token_tile(j / MTd);
      jb.w = G.gsdn + (size_t)jb.m * (Is / 64) * GEMM_BLK8; jb.int8 = 1; jb.ktiles = Is / 64;
      jb.bmap = CM_HS; jb.lomap = CM_HSLO; jb.gmap = CM_GHS;
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
  return __ldcg(g.S.groups + (j % ngroups));
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
  uint64_t full[NSG_MAX], empty[NSG_MAX], a_ready[NT_MAX], a_free[NT_MAX];
  uint64_t bb_full[2], acc_full[2], acc_free[2];   // per job parity
  uint64_t fold_sync;   // the four epilogue warps meet here (a bounded wait)
  uint32_t tslot;
  int ngroups, tw;      // the launch's row-tile count and token-tile width, read once
  volatile int abort;
};
static_assert(sizeof(Bars) <= S_BYTES - S_BAR, "barrier area");

// debug stamps (CTA 0, first 64 K-tiles): events 0 producer issued, 1 dequant saw the stage, 2 dequant done,
// 3 MMA issued, 4 epilogue saw the accumulator (at the job's last K-tile), 5 epilogue read it, 6 MMA saw A ready
// (only the traced instantiation of the kernel, TR = true, carries them: every instruction of the MMA warp's
// per-K-tile loop is on the pipeline's critical path)
#define GSTAMP(ev, k) do { if (TR && blockIdx.x == 0 && (k) < 64) g.trace[(ev) * 64 + (k)] = clock64(); } while (0)

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

// rows of a TMA box for a job of N rows (boxes of 16, 32 or 64)
__device__ __forceinline__ int box_of(int n) { return n <= 16 ? 0 : n <= 32 ? 1 : 2; }

template <bool TR>
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
      mbar_init(&bar->empty[s], 4 + 1);     // dequant warps (stage read) + MMA commit (B read)
    }
    for (int i = 0; i < NT_MAX; ++i) {
      mbar_init(&bar->a_ready[i], 4);
      mbar_init(&bar->a_free[i], 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&bar->bb_full[p], 1);       // the issuing producer's expect-tx arrival
      mbar_init(&bar->acc_full[p], 1);      // the MMA issuer's commit after the job's bias MMA
      mbar_init(&bar->acc_free[p], 4);      // the epilogue warps
    }
    mbar_init(&bar->fold_sync, 4);
    bar->abort = 0;
  }
  if (warp == 1) { tmem_alloc(&bar->tslot, 512); tmem_relinquish(); }
  // programmatic-dependent launch: everything above overlaps the previous kernel; from here on its outputs are
  // read (the bucketing's tile list, the activations)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    // phase 1 tiles the tokens 64 at a time; phases 2 and 3 take the bucketing's row tiles, and phase 3 tiles
    // the shared down's tokens as wide as the widest row tile, so no job is wider than that
    bar->ngroups = g.phase == 1 ? 0 : __ldcg(g.S.ctl);
    bar->tw = g.phase == 1 ? CHUNK_NT : min(CHUNK_NT, max(16, (__ldcg(g.S.ctl + 1) + 15) & ~15));
    fence_mbar_init();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tslot;
  const Geo geo = geo_of(g.phase);
  const uint32_t NSG = (uint32_t)geo.nsg;
  const int ngroups = bar->ngroups, tw = bar->tw;
  // tensor memory: accumulators (job parity) of dcols columns: aw for the sum (aw = the widest job's N rounded
  // up to 32), in phase 3 aw more for the low halves; the bias A operands (job parity, 32 columns: column g
  // holds the pair (b_g, b_g)); the A slots (64 columns: A1 | A2)
  const bool lo_phase = g.phase == 3;
  // the widest job: phase 1 token tiles of up to CHUNK_NT; phase 2 the expert row tiles (tw) and the shared
  // gate/up token tiles of up to CHUNK_NT; phase 3 tw
  const int tok_w = (min(g.T, CHUNK_NT) + 15) & ~15;
  const uint32_t aw = (uint32_t)(((g.phase == 1 ? tok_w : g.phase == 2 ? max(tw, tok_w) : tw) + 31) & ~31);
  const uint32_t dcols = lo_phase ? 2 * aw : aw, tlo = aw, ab0 = 2 * dcols, a0 = ab0 + 64;
  const int nt = min(NT_MAX, (int)((512 - a0) / 64));

  if (warp == 0 || warp >= WEP + 4) {
    // ------------------------------------------------------------------ producers
    // Producer p fills the stages of the K-tiles gk with gk % NPR == p, stepping NPR K-tiles at a time across
    // job boundaries. The whole warp walks, so every copy operand is warp-uniform, and one elected lane arms
    // the stage and issues its copies: the weight block (1-D bulk copy), then B hi and B lo (tensor loads).
    const uint32_t par = warp == 0 ? 0u : (uint32_t)(warp - WEP - 3);   // 0, 1, 2
    uint32_t gk = 0, njob = 0;   // position in the CTA's K-tile sequence; index of the current job
    // test hook: CTA 0 never arms or fills the stage of its first K-tile, so the roles waiting for it time
    // out and the CTA aborts
    const bool withhold = g.skip && blockIdx.x == 0;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sr;
    int kt = 0;
    bool have = job_next(g, it, jb);
    auto step = [&](int n) {
      kt += n;
      gk += (uint32_t)n;
      sr.adv(n, (int)NSG);
      while (have && kt >= jb.ktiles) {
        kt -= jb.ktiles;
        ++njob;
        have = job_next(g, it, jb);
      }
    };
    step((int)par);
    while (have) {
      const int blk = jb.int8 ? GEMM_BLK8 : GEMM_BLK4;
      const int box = box_of(jb.n);
      const bool lo = jb.lomap >= 0;
      const uint32_t pb = njob & 1u;
      // the job's bias tile, by the producer of its first K-tile, once the bias MMA of job njob - 2 (same
      // buffer) has completed
      if (kt == 0) {
        const bool ok = njob < 2 || wait(&bar->acc_full[pb], ((njob >> 1) - 1) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        if (elect_one()) {
          mbar_expect_tx(&bar->bb_full[pb], (16u << box) * 128u);
          tma_load_2d(smem + S_BB + pb * BB_BYTES, &g.maps.m[jb.gmap][box], 0, jb.row0, &bar->bb_full[pb]);
        }
        __syncwarp();
      }
      const int s = sr.t;
      const bool ok = gk < NSG || wait(&bar->empty[s], sr.ph ^ 1u);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      if (!(withhold && gk == 0)) {
        uint8_t* st = smem + s * geo.bytes;
        if (elect_one()) {
          mbar_expect_tx(&bar->full[s], (uint32_t)blk + (16u << box) * 128u * (lo ? 2u : 1u));
          const int kg = jb.k0 + kt;   // K-tile within the band
          bulk_g2s(st + ST_W, jb.w + (size_t)kg * blk, (uint32_t)blk, &bar->full[s]);
          tma_load_2d(st + geo.bhi, &g.maps.m[jb.bmap][box], kg * 64, jb.row0, &bar->full[s]);
          if (lo) tma_load_2d(st + geo.blo, &g.maps.m[jb.lomap][box], kg * 64, jb.row0, &bar->full[s]);
          GSTAMP(0, gk);
        }
        __syncwarp();
      }
      step(NPR);
    }
    // drain: every copy this warp issued must have landed before the CTA leaves (the withheld one was never
    // issued); only the last NSG K-tiles can still be in flight, and of the bias tiles those of the last two
    // jobs (whichever producer issued them; after an abort the waits give up at once)
    if (lane == 0) {
      const uint32_t cnt = gk < (uint32_t)NSG ? gk : (uint32_t)NSG;
      for (uint32_t q = gk - cnt; q < gk; ++q)
        if (q % NPR == par && !(withhold && q == 0)) mbar_wait(&bar->full[q % NSG], (q / NSG) & 1u, to);
    }
    for (uint32_t j = njob >= 2 ? njob - 2 : 0; j < njob; ++j) (void)wait(&bar->bb_full[j & 1u], (j >> 1) & 1u);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    // The whole warp steps through the loop and waits, so the descriptors and TMEM addresses are warp-uniform;
    // one elected lane (the same one every time) issues the MMAs and the commits.
    uint32_t gk = 0, njob = 0;
    bool run = true;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sl, sr;
    // B descriptors of stage 0 and of bias tile 0; a stage (bias tile) further on adds its byte offset / 16 to
    // the start-address field (shared-memory addresses stay below 256 KB, so the field never carries)
    const uint64_t dh0 = umma_desc_sw128(smem_u32(smem + geo.bhi)), dl0 = umma_desc_sw128(smem_u32(smem + geo.blo));
    const uint64_t db0 = umma_desc_sw128(smem_u32(smem + S_BB));
    const uint32_t sstep = (uint32_t)geo.bytes >> 4;
    const uint32_t dh_lo = (uint32_t)dh0, dh_hi = (uint32_t)(dh0 >> 32), dl_lo = (uint32_t)dl0, dl_hi = (uint32_t)(dl0 >> 32);
    while (run && job_next(g, it, jb)) {
      const uint32_t idesc = umma_idesc_f16(128, jb.n);
      const bool lo = jb.lomap >= 0;
      const uint32_t pb = njob & 1u, d = tmem + pb * dcols, ab = tmem + ab0 + 32u * pb;
      // the job accumulates in accumulator pb, which the epilogue of job njob - 2 must have read
      {
        const bool ok = njob < 2 || wait(&bar->acc_free[pb], ((njob >> 1) - 1) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      // two K-tiles per pass where the job has them: one vote and one fence for both
      for (int kt = 0; kt < jb.ktiles;) {
        const int n2 = kt + 1 < jb.ktiles ? 2 : 1;
        SlotRing sl1 = sl, sr1 = sr;
        sl1.next(nt);
        sr1.next(NSG);
        // a_ready implies full[s] (the dequantisation waited for it)
        // both probes issued back to back (their latencies overlap); the bounded waits only if one is not ready
        const bool r0 = mbar_try_wait(&bar->a_ready[sl.t], sl.ph);
        const bool r1 = n2 == 2 ? mbar_try_wait(&bar->a_ready[sl1.t], sl1.ph) : true;
        bool ok = r0 && r1;
        if (!ok) ok = (r0 || wait(&bar->a_ready[sl.t], sl.ph)) && (r1 || wait(&bar->a_ready[sl1.t], sl1.ph));
        const bool last = kt + n2 == jb.ktiles;
        if (last) ok = ok && wait(&bar->bb_full[pb], (njob >> 1) & 1u);
        if (!__all_sync(0xFFFFFFFFu, ok)) { run = false; break; }
        tc_fence_after();
        // B descriptors of the stages; a K step of 16 elements advances the start address by 32 bytes (2 units)
        const uint32_t so0 = (uint32_t)sr.t * sstep, so1 = (uint32_t)sr1.t * sstep;
        const uint32_t a0t = tmem + a0 + 64u * (uint32_t)sl.t, a1t = tmem + a0 + 64u * (uint32_t)sl1.t;
        if (elect_one()) {
          GSTAMP(6, gk);
          // D += A1 B + A2 B: the exact products s q x; then the low halves' D_lo += A1 B_lo
          umma_f16_ktile<true>(d, a0t, dh_lo + so0, dh_hi, idesc, kt > 0 ? 1u : 0u);
          if (lo) umma_f16_ktile<false>(d + tlo, a0t, dl_lo + so0, dl_hi, idesc, kt > 0 ? 1u : 0u);
          umma_commit(&bar->empty[sr.t]);
          umma_commit(&bar->a_free[sl.t]);
          if (n2 == 2) {
            umma_f16_ktile<true>(d, a1t, dh_lo + so1, dh_hi, idesc, 1u);
            if (lo) umma_f16_ktile<false>(d + tlo, a1t, dl_lo + so1, dl_hi, idesc, 1u);
            umma_commit(&bar->empty[sr1.t]);
            umma_commit(&bar->a_free[sl1.t]);
          }
          if (last) {
            // the offset term: D += (b_g, b_g) . (sum_hi_g, sum_lo_g) over the job's groups, 8 groups per
            // K step; the bias columns past the job's groups are zero
            const int nbk = (jb.ktiles + 7) >> 3, kb0 = jb.k0 >> 3;   // k0: a multiple of 8 groups
            const uint64_t bb = db0 + (uint64_t)(pb * (BB_BYTES >> 4));
            for (int ks = 0; ks < nbk; ++ks) umma_f16_ts(d, ab + 8 * ks, bb + 2 * (kb0 + ks), idesc, 1u);
            umma_commit(&bar->acc_full[pb]);
          }
          GSTAMP(3, gk);
        }
        if (n2 == 2) {
          sl = sl1;
          sr = sr1;
        }
        sl.next(nt);
        sr.next(NSG);
        gk += (uint32_t)n2;
        kt += n2;
      }
      ++njob;
    }
    // the last MMAs must have completed before TMEM is released (a commit tracks all earlier MMAs of its thread)
    if (lane == 0 && gk > 0) mbar_wait(&bar->empty[(gk - 1) % NSG], ((gk - 1) / NSG) & 1u, to);
    __syncwarp();
  } else if (warp < WEP) {
    // ------------------------------------------------------------------ dequantise
    const int grp = (warp - 2) >> 2;          // this group takes the K-tiles gk with gk % NDQ == grp
    const int r = (warp & 3) * 32 + lane;     // band row = the TMEM lane this warp may access
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const __half2 k1024 = __float2half2_rn(1024.0f), k16 = __float2half2_rn(0.0625f), k64 = __float2half2_rn(-64.0f);
    uint32_t gk = 0, njob = 0;
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    SlotRing sl, sr;
    // the walk steps NDQ K-tiles at a time, crossing job boundaries as it goes
    int kt = 0;
    bool have = job_next(g, it, jb);
    auto step = [&](int n) {
      kt += n;
      gk += (uint32_t)n;
      sl.adv(n, nt);
      sr.adv(n, (int)NSG);
      while (have && kt >= jb.ktiles) {
        kt -= jb.ktiles;
        ++njob;
        have = job_next(g, it, jb);
      }
    };
    step(grp);
    while (have) {
      {
        const uint32_t pb = njob & 1u, tab = trow + ab0 + 32u * pb;
        const int s = sr.t, t = sl.t;
        // the stage landed; A slot t is free (the MMAs of K-tile gk - nt completed); the bias columns of
        // parity pb are free (the bias MMA of job njob - 2 completed)
        if ((gk >= NSG && !wait(&bar->empty[s], sr.ph ^ 1u)) || !wait(&bar->full[s], sr.ph) ||
            (gk >= (uint32_t)nt && !wait(&bar->a_free[t], sl.ph ^ 1u)) ||
            (njob >= 2 && !wait(&bar->acc_full[pb], ((njob >> 1) - 1) & 1u)))
          break;
        tc_fence_after();
        if (r == 0) GSTAMP(1, gk);
        const uint8_t* st = smem + s * geo.bytes + ST_W;
        // row r's (s, b) pair
        const uint32_t sbw = *reinterpret_cast<const uint32_t*>(st + 128 * (jb.int8 ? 64 : 32) + r * 4);
        const __half2 s2 = __low2half2(*reinterpret_cast<const __half2*>(&sbw));
        // row r of A1 and A2 in K order: column 4c + k holds the pair k of 8-column block c. A1 = fp16(s q),
        // A2 = s q - A1 (exact: the residual of rounding s q, a multiple of s's unit in the last place with at
        // most 19 significant bits, has at most 9 and is a multiple of that unit, never below 2^-24). Two
        // halves of 16 columns, each stored as soon as it is made.
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
        // the K-tile's bias column (b, b); the first K-tile also zeroes the columns past the job's groups up to
        // the bias MMA's K extent (8 groups per K step)
        {
          const uint32_t bpair = (sbw >> 16) | (sbw & 0xFFFF0000u);
          tmem_st1(tab + (uint32_t)kt, bpair);
          if (kt == 0)
            for (int c = jb.ktiles; c < ((jb.ktiles + 7) & ~7); ++c) tmem_st1(tab + (uint32_t)c, 0u);
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
      step(NDQ);
    }
  } else if (warp < WEP + 4) {
    // ------------------------------------------------------------------ epilogue
    const int q4 = warp & 3;               // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;          // band row
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    float* ep = reinterpret_cast<float*>(smem + S_EP);      // [128 rows][65] the job's accumulator
    const GemmLayout& G = g.G;
    const ChunkScratch& S = g.S;
    uint32_t fph = 0, njob = 0, gk = 0;
    // the four epilogue warps meet (bounded: a warp that has aborted makes the others time out, never hang)
    auto fold_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->fold_sync);
      const bool ok = wait(&bar->fold_sync, fph);
      fph ^= 1u;
      return ok;
    };
    JobIter it;
    job_begin(g, ngroups, tw, it);
    Job jb;
    while (job_next(g, it, jb)) {
      const uint32_t pb = njob & 1u;
      gk += (uint32_t)jb.ktiles;
      if (!wait(&bar->acc_full[pb], (njob >> 1) & 1u)) break;
      tc_fence_after();
      if (r == 0) GSTAMP(4, gk - 1);
      // the accumulator (+ the low halves' share / 4096) goes to shared memory, 16 columns at a time
      const uint32_t d = trow + pb * dcols;
#pragma unroll 1
      for (int c0 = 0; c0 < jb.n; c0 += 16) {
        uint32_t v[16];
        tmem_ld16_nowait(d + c0, v);
        tmem_wait_ld(v);
        if (jb.lomap >= 0) {
          uint32_t w[16];
          tmem_ld16_nowait(d + tlo + c0, w);
          tmem_wait_ld(w);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ep[r * 65 + c0 + i] = fmaf(__uint_as_float(w[i]), 1.0f / 4096.0f, __uint_as_float(v[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) ep[r * 65 + c0 + i] = __uint_as_float(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->acc_free[pb]);
      if (r == 0) GSTAMP(5, gk - 1);
      ++njob;
      if (!fold_sync()) break;
      const int cnt = jb.cnt;
      if (jb.kind == GK_ROUTER) {
        // thread = band row (router output row), tokens in a loop; consecutive rows on consecutive lanes
        const int er = jb.m * 128 + r;
        if (er <= G.E)
#pragma unroll 4
          for (int i = 0; i < cnt; ++i)
            S.logits[((size_t)jb.part * g.T + jb.row0 + i) * logit_stride(G.E) + er] = ep[r * 65 + i];
      } else if (jb.kind == GK_SHDN || jb.kind == GK_EXDN) {
        float* dst = jb.kind == GK_SHDN ? S.ys : S.y;
#pragma unroll 4
        for (int i = 0; i < cnt; ++i) dst[(size_t)(jb.row0 + i) * G.H + jb.m * 128 + r] = ep[r * 65 + i];
      } else {
        // SwiGLU: rows 0-63 are gate units 64m.., rows 64-127 the matching up units. h = silu(g) * u is split
        // into fp16 hi + lo/4096 halves, the down projection's B operand; the 64 units are group m of the down
        // projection's reduction, so the group's sum (of hi + lo/4096, the values the MMAs see) goes into the
        // row's group-sum entries 2m, 2m + 1. Warp = token (4 at a time), lane = units u and u + 32.
        const bool sh = jb.kind == GK_SHGU;
        const int kd = sh ? G.Is : G.I;
        uint16_t* dhi = sh ? S.hs : S.hh;
        uint16_t* dlo = sh ? S.hs_lo : S.hh_lo;
        uint16_t* gsum = sh ? S.gs_hs : S.gs_hh;
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
          if (lane == 0) {
            const __half phi = __float2half_rn(part);
            const __half plo = __float2half_rn(part - __half2float(phi));
            *reinterpret_cast<uint32_t*>(gsum + (size_t)(jb.row0 + i) * GSUM_COLS + 2 * jb.m) =
                (uint32_t)__half_as_ushort(phi) | ((uint32_t)__half_as_ushort(plo) << 16);
          }
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
      e = cudaFuncSetAttribute(k_chunk_gemm<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_chunk_gemm<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  // programmatic-dependent: the CTAs set up their barriers and tensor memory while the previous kernel ends
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(GTH);
  cfg.dynamicSmemBytes = GEMM_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return g.trace ? cudaLaunchKernelEx(&cfg, k_chunk_gemm<true>, g) : cudaLaunchKernelEx(&cfg, k_chunk_gemm<false>, g);
}

}  // namespace moe
