// C ABI of the block (declared in include/moe_block.h): argument validation, device memory, weight loading
// and dispatch to the kernels. No call throws or aborts; every failure is a negative status.
#include <cuda_runtime.h>
#include <new>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/moe_block.h"
#include "chunk.cuh"
#include "decode.cuh"
#include "layout.cuh"
#include "repack.cuh"

using namespace moe;

struct moe_block {
  moe_block_config_t cfg;
  MoeLayout L;
  int dev = 0, num_sms = 0, max_smem = 0;
  uint8_t* wstore = nullptr;                       // one allocation for all repacked weights
  uint8_t *router = nullptr, *sh_gu = nullptr, *sh_dn = nullptr, *ex_gu = nullptr, *ex_dn = nullptr;
  uint16_t* gamma = nullptr;
  bool loaded = false, has_gamma = false;
  int dec_T = 0;                                   // largest T the decode scratch holds
  float *logits = nullptr, *hs = nullptr, *hbuf = nullptr;
  uint64_t* xlog = nullptr;
  uint32_t *counters = nullptr, *status = nullptr;
  int32_t* rec_ids = nullptr;
  float *rec_w = nullptr, *rec_sg = nullptr;
  uint16_t *xbuf = nullptr, *obuf = nullptr;       // staging for forward_host
  uint32_t* status_host = nullptr;                 // pinned copy of the status word (forward_host)
  uint64_t timeout_ns = 500ull * 1000 * 1000;
  int skip_arrive = 0;
  int last_launches = 0;
  int last_T = 0;
  DecodeLaunch plans[DEC_TMAX + 1];                // launch plan per T, computed at create
  bool has_dec1 = false;                           // the single-token kernel serves T = 1
  Decode1Launch plan1;
  cudaStream_t last_stream = nullptr;              // stream of the last forward call (for get_status)
  uint64_t* trace = nullptr;                       // optional phase-timestamp buffer (debug)
  // prompt-chunk path (T > 16): GEMM-layout weight copy and its scratch, only when max_tokens > 16
  bool chunk = false;
  uint8_t* gstore = nullptr;
  uint8_t* cscratch = nullptr;
  GemmLayout G;
  ChunkScratch CS;
  ChunkMaps maps;
};

static thread_local char g_cuda_err[256] = "";

static int cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}
#define CK(call)                                        \
  do {                                                  \
    cudaError_t _e = (call);                            \
    if (_e != cudaSuccess) return cuda_fail(_e, #call); \
  } while (0)

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

extern "C" const char* moe_last_cuda_error(void) { return g_cuda_err; }

extern "C" const char* moe_block_strerror(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_NOT_LOADED: return "weights not loaded";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case MOE_ERR_NO_DEVICE: return "no sm_103 device";
    default: return "unknown status";
  }
}

static void free_all(moe_block* b) {
  cudaFree(b->wstore);
  cudaFree(b->gamma);
  cudaFree(b->logits);
  cudaFree(b->xlog);
  cudaFree(b->hs);
  cudaFree(b->hbuf);
  cudaFree(b->counters);
  cudaFree(b->rec_ids);
  cudaFree(b->rec_w);
  cudaFree(b->rec_sg);
  cudaFree(b->xbuf);
  cudaFree(b->obuf);
  cudaFree(b->gstore);
  cudaFree(b->cscratch);
  cudaFreeHost(b->status_host);
}

// the shapes the library has kernels for (MOE_OK) or not (MOE_ERR_UNSUPPORTED)
static int check_config(const moe_block_config_t& c) {
  if (c.group_size != 64) return MOE_ERR_UNSUPPORTED;
  if (c.hidden != 512 && c.hidden != 1024 && c.hidden != 2048) return MOE_ERR_UNSUPPORTED;
  if (c.n_experts < 1 || c.n_experts > 512) return MOE_ERR_UNSUPPORTED;
  if (c.top_k < 1 || c.top_k > 16 || c.top_k > c.n_experts) return MOE_ERR_UNSUPPORTED;
  if (c.expert_inter < 64 || c.expert_inter > 1024 || c.expert_inter % 64) return MOE_ERR_UNSUPPORTED;
  if (c.shared_inter < 64 || c.shared_inter > 1024 || c.shared_inter % 64) return MOE_ERR_UNSUPPORTED;
  if (c.max_tokens < 1 || c.max_tokens > 4096) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

extern "C" int moe_debug_decode_plan(const moe_block_config_t* cfg, int T, int num_sms, int max_smem,
                                     int32_t* out) {
  if (!cfg || !out || T < 1 || num_sms < 1 || max_smem < 1) return MOE_ERR_INVALID_ARG;
  const int st = check_config(*cfg);
  if (st != MOE_OK) return st;
  const MoeLayout L = moe_make_layout(cfg->hidden, cfg->n_experts, cfg->top_k, cfg->expert_inter,
                                      cfg->shared_inter);
  if (!decode_supported(L)) return MOE_ERR_UNSUPPORTED;
  DecodeLaunch pl;
  if (!decode_plan(L, T, num_sms, max_smem, &pl)) return MOE_ERR_UNSUPPORTED;
  out[0] = pl.grid;
  out[1] = pl.smem;
  out[2] = pl.NS;
  out[3] = pl.SS;
  out[4] = pl.hp;
  return MOE_OK;
}

extern "C" int moe_block_create(const moe_block_config_t* cfg, moe_block_t** out) {
  if (!cfg || !out) return MOE_ERR_INVALID_ARG;
  const moe_block_config_t c = *cfg;
  {
    const int st = check_config(c);
    if (st != MOE_OK) return st;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_NO_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) {
    snprintf(g_cuda_err, sizeof(g_cuda_err), "device is sm_%d%d, library is built for sm_103a", prop.major,
             prop.minor);
    return MOE_ERR_NO_DEVICE;
  }
  moe_block* b = new (std::nothrow) moe_block;
  if (!b) return MOE_ERR_CUDA;
  b->cfg = c;
  b->L = moe_make_layout(c.hidden, c.n_experts, c.top_k, c.expert_inter, c.shared_inter);
  b->dev = dev;
  b->num_sms = prop.multiProcessorCount;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  b->max_smem = optin;
  // the decode kernel needs a plan for every T it may see
  if (!decode_supported(b->L)) { delete b; return MOE_ERR_UNSUPPORTED; }
  b->dec_T = c.max_tokens < DEC_TMAX ? c.max_tokens : DEC_TMAX;
  for (int T = 1; T <= b->dec_T; ++T) {
    if (!decode_plan(b->L, T, b->num_sms, b->max_smem, &b->plans[T])) { delete b; return MOE_ERR_UNSUPPORTED; }
  }
  b->has_dec1 = decode1_plan(b->L, b->num_sms, b->max_smem, &b->plan1);
  // the grid-wide counts of the decode kernels need every CTA of a launch resident at once: refuse a device
  // on which the grid does not fit
  {
    int per_sm = 0;
    if (b->has_dec1) {
      if (decode1_occupancy(b->L, b->plan1, &per_sm) != cudaSuccess || per_sm * b->num_sms < b->plan1.grid)
        b->has_dec1 = false;
    }
    for (int T = 1; T <= b->dec_T; ++T) {
      per_sm = 0;
      const cudaError_t oe = decode_occupancy(b->L, b->plans[T], &per_sm);
      if (oe != cudaSuccess || per_sm * b->num_sms < b->plans[T].grid) {
        const int grid = b->plans[T].grid;
        delete b;
        if (oe != cudaSuccess) return cuda_fail(oe, "decode occupancy");
        snprintf(g_cuda_err, sizeof(g_cuda_err), "the decode grid of %d CTAs does not fit the device at once",
                 grid);
        return MOE_ERR_UNSUPPORTED;
      }
    }
  }
  const MoeLayout& L = b->L;
  size_t total = L.router_bytes + L.shgu_bytes + L.shdn_bytes + L.exgu_bytes + L.exdn_bytes;
  cudaError_t e = cudaMalloc(&b->wstore, total);
  if (e == cudaSuccess) {
    b->router = b->wstore;
    b->sh_gu = b->router + L.router_bytes;
    b->sh_dn = b->sh_gu + L.shgu_bytes;
    b->ex_gu = b->sh_dn + L.shdn_bytes;
    b->ex_dn = b->ex_gu + L.exgu_bytes;
  }
  const int T = b->dec_T;
  if (e == cudaSuccess) e = cudaMalloc(&b->gamma, (size_t)c.hidden * 2);
  if (e == cudaSuccess) e = cudaMalloc(&b->logits, (size_t)T * (c.n_experts + 1) * 4);
  // tags start at 0 and the first launch publishes epoch 1, so nothing stale is ever taken for fresh
  if (e == cudaSuccess) e = cudaMalloc(&b->xlog, XLOG_COPIES * xlog_stride(c.n_experts) * 8);
  if (e == cudaSuccess) e = cudaMemset(b->xlog, 0, XLOG_COPIES * xlog_stride(c.n_experts) * 8);
  if (e == cudaSuccess) e = cudaMalloc(&b->hs, (size_t)T * c.shared_inter * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->hbuf, decode_hbuf_floats(L, T) * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->counters, CNT_WORDS * 4);
  if (e == cudaSuccess) e = cudaMemset(b->counters, 0, CNT_WORDS * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->rec_ids, (size_t)c.max_tokens * c.top_k * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->rec_w, (size_t)c.max_tokens * c.top_k * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->rec_sg, (size_t)c.max_tokens * 4);
  if (e == cudaSuccess) e = cudaMalloc(&b->xbuf, (size_t)c.max_tokens * c.hidden * 2);
  if (e == cudaSuccess) e = cudaMalloc(&b->obuf, (size_t)c.max_tokens * c.hidden * 2);
  if (e == cudaSuccess) e = cudaHostAlloc(&b->status_host, 16, cudaHostAllocDefault);
  if (e == cudaSuccess) *b->status_host = 0;
  if (e == cudaSuccess && c.max_tokens > DEC_TMAX) {
    b->chunk = true;
    e = cudaMalloc(&b->gstore, gemm_store_bytes(L));
    if (e == cudaSuccess) e = cudaMalloc(&b->cscratch, chunk_scratch_bytes(L, c.max_tokens));
    // zero once: the group-sum rows' entries past the matrices' groups stay zero (the GEMM multiplies them)
    if (e == cudaSuccess) e = cudaMemset(b->cscratch, 0, chunk_scratch_bytes(L, c.max_tokens));
    if (e == cudaSuccess) {
      b->G = gemm_layout_carve(L, b->gstore);
      b->CS = chunk_scratch_carve(L, c.max_tokens, b->cscratch);
      e = chunk_make_maps(L, b->CS, c.max_tokens, &b->maps);
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(b);
    delete b;
    return cuda_fail(e, "moe_block_create");
  }
  b->status = b->counters + CNT_STATUS;
  *out = b;
  return MOE_OK;
}

extern "C" void moe_block_destroy(moe_block_t* b) {
  if (!b) return;
  cudaDeviceSynchronize();
  free_all(b);
  delete b;
}

extern "C" int moe_block_load_affine(moe_block_t* b, const moe_affine_weights_t* src, void* stream) {
  if (!b || !src) return MOE_ERR_INVALID_ARG;
  moe_block_weights_t w;
  const int st = moe_affine_convert(&b->cfg, src, &w);
  if (st != MOE_OK) return st;
  const int r = moe_block_load_weights(b, &w, 0, stream);
  moe_affine_free(&w);
  return r;
}

extern "C" int moe_block_load_weights(moe_block_t* b, const moe_block_weights_t* w, int on_device, void* stream) {
  if (!b || !w) return MOE_ERR_INVALID_ARG;
  const void* req[] = {w->router_q, w->router_s, w->router_b, w->exp_gate_q, w->exp_gate_s, w->exp_gate_b,
                       w->exp_up_q, w->exp_up_s, w->exp_up_b, w->exp_down_q, w->exp_down_s, w->exp_down_b,
                       w->sh_gate_q, w->sh_gate_s, w->sh_gate_b, w->sh_up_q, w->sh_up_s, w->sh_up_b,
                       w->sh_down_q, w->sh_down_s, w->sh_down_b};
  for (const void* p : req)
    if (!p) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const moe_block_config_t& c = b->cfg;
  const size_t H = c.hidden, E = c.n_experts, I = c.expert_inter, Is = c.shared_inter;
  // sizes in bytes of the 21 canonical arrays, in the order of `req`
  const size_t sz[] = {(E + 1) * H, (E + 1) * (H / 64) * 2, (E + 1) * (H / 64) * 2,
                       E * I * H / 2, E * I * (H / 64) * 2, E * I * (H / 64) * 2,
                       E * I * H / 2, E * I * (H / 64) * 2, E * I * (H / 64) * 2,
                       E * H * I / 2, E * H * (I / 64) * 2, E * H * (I / 64) * 2,
                       Is * H, Is * (H / 64) * 2, Is * (H / 64) * 2,
                       Is * H, Is * (H / 64) * 2, Is * (H / 64) * 2,
                       H * Is, H * (Is / 64) * 2, H * (Is / 64) * 2};
  const void* dptr[21];
  uint8_t* tmp = nullptr;
  if (on_device) {
    for (int i = 0; i < 21; ++i) dptr[i] = req[i];
  } else {
    size_t total = 0;
    for (size_t s : sz) total += (s + 255) & ~(size_t)255;
    CK(cudaMalloc(&tmp, total));
    size_t off = 0;
    for (int i = 0; i < 21; ++i) {
      cudaError_t e = cudaMemcpyAsync(tmp + off, req[i], sz[i], cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) { cudaFree(tmp); return cuda_fail(e, "load_weights copy"); }
      dptr[i] = tmp + off;
      off += (sz[i] + 255) & ~(size_t)255;
    }
  }
  RepackSrc src;
  src.router_q = (const uint8_t*)dptr[0]; src.router_s = (const uint16_t*)dptr[1]; src.router_b = (const uint16_t*)dptr[2];
  src.exp_gate_q = (const uint8_t*)dptr[3]; src.exp_gate_s = (const uint16_t*)dptr[4]; src.exp_gate_b = (const uint16_t*)dptr[5];
  src.exp_up_q = (const uint8_t*)dptr[6]; src.exp_up_s = (const uint16_t*)dptr[7]; src.exp_up_b = (const uint16_t*)dptr[8];
  src.exp_down_q = (const uint8_t*)dptr[9]; src.exp_down_s = (const uint16_t*)dptr[10]; src.exp_down_b = (const uint16_t*)dptr[11];
  src.sh_gate_q = (const uint8_t*)dptr[12]; src.sh_gate_s = (const uint16_t*)dptr[13]; src.sh_gate_b = (const uint16_t*)dptr[14];
  src.sh_up_q = (const uint8_t*)dptr[15]; src.sh_up_s = (const uint16_t*)dptr[16]; src.sh_up_b = (const uint16_t*)dptr[17];
  src.sh_down_q = (const uint8_t*)dptr[18]; src.sh_down_s = (const uint16_t*)dptr[19]; src.sh_down_b = (const uint16_t*)dptr[20];
  RepackDst dst{b->router, b->sh_gu, b->sh_dn, b->ex_gu, b->ex_dn};
  cudaError_t e = repack_all(src, b->L, dst, st);
  // the repack's scale-range flag: a spare word of the chunk scratch's control block
  uint32_t* range_bad = b->chunk ? reinterpret_cast<uint32_t*>(b->CS.ctl) + 8 : nullptr;
  if (e == cudaSuccess && b->chunk) e = gemm_repack(src, b->G, range_bad, st);
  if (e == cudaSuccess && w->rms_gamma) {
    e = cudaMemcpyAsync(b->gamma, w->rms_gamma, H * 2, on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                        st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (tmp) cudaFree(tmp);
  if (e != cudaSuccess) return cuda_fail(e, "moe_block_load_weights");
  if (b->chunk) {
    uint32_t bad = 0;
    e = cudaMemcpy(&bad, range_bad, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "moe_block_load_weights");
    if (bad) {
      b->loaded = false;
      return MOE_ERR_INVALID_ARG;
    }
  }
  b->has_gamma = w->rms_gamma != nullptr;
  b->loaded = true;
  return MOE_OK;
}

static DecodeArgs decode_args(moe_block* b, const uint16_t* x, uint16_t* out, uint16_t* out2, int T, int t0,
                              const uint16_t* gamma, float eps) {
  DecodeArgs a;
  a.router = b->router; a.sh_gu = b->sh_gu; a.sh_dn = b->sh_dn; a.ex_gu = b->ex_gu; a.ex_dn = b->ex_dn;
  a.x = x + (size_t)t0 * b->cfg.hidden;
  a.out = out + (size_t)t0 * b->cfg.hidden;
  a.out2 = out2 ? out2 + (size_t)t0 * b->cfg.hidden : nullptr;
  a.gamma = gamma;
  a.eps = eps;
  a.T = T;
  a.logits = b->logits; a.xlog = b->xlog; a.hs = b->hs; a.hbuf = b->hbuf;
  a.counters = b->counters; a.status = b->status;
  a.rec_ids = b->rec_ids + (size_t)t0 * b->cfg.top_k;
  a.rec_w = b->rec_w + (size_t)t0 * b->cfg.top_k;
  a.rec_sg = b->rec_sg + t0;
  a.timeout_ns = b->timeout_ns;
  a.skip_arrive = b->skip_arrive;
  a.trace = b->trace;
  b->skip_arrive = 0;
  return a;
}

static int run_forward(moe_block* b, const uint16_t* x, uint16_t* out, int T, const uint16_t* gamma, float eps,
                       cudaStream_t st, uint16_t* out2 = nullptr) {
  b->last_launches = 0;
  b->last_T = T;
  b->last_stream = st;
  if (T == 1 && b->has_dec1) {
    cudaError_t e = decode1_launch(b->L, decode_args(b, x, out, out2, 1, 0, gamma, eps), b->plan1, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    b->last_launches = 1;
    return MOE_OK;
  }
  if (T > DEC_TMAX && b->chunk) {
    int n = 0;
    cudaError_t e = chunk_forward(b->L, b->G, b->CS, b->maps, b->cfg.max_tokens, b->num_sms, x, out, T, gamma, eps,
                                  b->rec_ids, b->rec_w,
                                  b->rec_sg, b->status, b->timeout_ns, b->trace, st, &n, b->skip_arrive);
    b->skip_arrive = 0;
    b->last_launches = n;
    if (e != cudaSuccess) return cuda_fail(e, "chunk forward");
    return MOE_OK;
  }
  for (int t0 = 0; t0 < T; t0 += DEC_TMAX) {
    const int n = T - t0 < DEC_TMAX ? T - t0 : DEC_TMAX;
    const DecodeLaunch& pl = b->plans[n];
    const DecodeArgs a = decode_args(b, x, out, out2, n, t0, gamma, eps);
    cudaError_t e = decode_launch(b->L, a, pl, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    ++b->last_launches;
  }
  return MOE_OK;
}

extern "C" int moe_block_forward(moe_block_t* b, const void* x, void* out, int T, void* stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > b->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) { b->last_launches = 0; return MOE_OK; }
  if (!x || !out || !aligned16(x) || !aligned16(out) || x == out) return MOE_ERR_INVALID_ARG;
  if (!b->loaded) return MOE_ERR_NOT_LOADED;
  return run_forward(b, (const uint16_t*)x, (uint16_t*)out, T, nullptr, 0.f, (cudaStream_t)stream);
}

extern "C" int moe_block_forward_residual(moe_block_t* b, const void* h_in, void* h_out, int T, float eps,
                                          void* stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > b->cfg.max_tokens || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) { b->last_launches = 0; return MOE_OK; }
  if (!h_in || !h_out || !aligned16(h_in) || !aligned16(h_out)) return MOE_ERR_INVALID_ARG;
  if (!b->loaded) return MOE_ERR_NOT_LOADED;
  if (!b->has_gamma) return MOE_ERR_NOT_LOADED;
  if (T > DEC_TMAX && h_in == h_out) return MOE_ERR_INVALID_ARG;
  return run_forward(b, (const uint16_t*)h_in, (uint16_t*)h_out, T, b->gamma, eps, (cudaStream_t)stream);
}

extern "C" int moe_block_forward_host(moe_block_t* b, const void* x_host, void* out_host, int T, void* stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > b->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (!b->loaded) return MOE_ERR_NOT_LOADED;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t bytes = (size_t)T * b->cfg.hidden * 2;
  CK(cudaMemcpyAsync(b->xbuf, x_host, bytes, cudaMemcpyHostToDevice, st));
  int s = run_forward(b, b->xbuf, b->obuf, T, nullptr, 0.f, st);
  if (s != MOE_OK) return s;
  CK(cudaMemcpyAsync(out_host, b->obuf, bytes, cudaMemcpyDeviceToHost, st));
  CK(cudaMemcpyAsync(b->status_host, b->status, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  // the call has completed: a bounded device wait that ran out is reported here (the handle's device state is
  // reset as in moe_block_get_status)
  if (*b->status_host) return moe_block_get_status(b, nullptr);
  return MOE_OK;
}

extern "C" int moe_block_get_status(moe_block_t* b, uint32_t* flags) {
  if (!b) return MOE_ERR_INVALID_ARG;
  // the handle's device work: everything issued to the stream of its last forward call
  CK(cudaStreamSynchronize(b->last_stream));
  uint32_t st = 0;
  CK(cudaMemcpy(&st, b->status, 4, cudaMemcpyDeviceToHost));
  if (flags) *flags = st;
  if (st) {
    // every count, the status word and the single-token epoch, and the published logit tags with it (the next
    // launch publishes epoch 1, which nothing left in the buffers carries)
    CK(cudaMemset(b->counters, 0, CNT_WORDS * 4));
    CK(cudaMemset(b->xlog, 0, XLOG_COPIES * xlog_stride(b->cfg.n_experts) * 8));
    CK(cudaDeviceSynchronize());
    if (b->status_host) *b->status_host = 0;
    return MOE_ERR_DEVICE_TIMEOUT;
  }
  return MOE_OK;
}

extern "C" int moe_block_debug_dequant(moe_block_t* b, int which, int index, float* out, void* stream) {
  if (!b || !out || which < 0 || which > 6) return MOE_ERR_INVALID_ARG;
  if (!b->loaded) return MOE_ERR_NOT_LOADED;
  if (which >= 1 && which <= 3 && (index < 0 || index >= b->cfg.n_experts)) return MOE_ERR_INVALID_ARG;
  const uint8_t* base = which == 0 ? b->router : which <= 2 ? b->ex_gu : which == 3 ? b->ex_dn
                      : which <= 5 ? b->sh_gu : b->sh_dn;
  cudaError_t e = debug_dequant(base, b->L, which, index, out, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "debug_dequant");
  return MOE_OK;
}

// Each token's k (id, weight) pairs of the routing record into ascending id order (the single-token kernel records
// them in selection order); one thread per token, insertion sort. Idempotent.
__global__ void k_sort_routing(int32_t* ids, float* w, int T, int K) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int32_t* id = ids + (size_t)t * K;
  float* wt = w + (size_t)t * K;
  for (int i = 1; i < K; ++i) {
    const int32_t ki = id[i];
    const float wi = wt[i];
    int j = i - 1;
    while (j >= 0 && id[j] > ki) {
      id[j + 1] = id[j];
      wt[j + 1] = wt[j];
      --j;
    }
    id[j + 1] = ki;
    wt[j + 1] = wi;
  }
}

extern "C" int moe_block_debug_last_routing(moe_block_t* b, int T, float* logits, int32_t* ids, float* w,
                                            float* sg, void* stream) {
  if (!b || T < 1 || T > b->last_T) return MOE_ERR_INVALID_ARG;
  if (logits && T > b->dec_T) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int E = b->cfg.n_experts, K = b->cfg.top_k;
  if (logits) CK(cudaMemcpyAsync(logits, b->logits, (size_t)T * (E + 1) * 4, cudaMemcpyDeviceToDevice, st));
  k_sort_routing<<<(T + 127) / 128, 128, 0, st>>>(b->rec_ids, b->rec_w, T, K);
  CK(cudaGetLastError());
  if (ids) CK(cudaMemcpyAsync(ids, b->rec_ids, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, st));
  if (w) CK(cudaMemcpyAsync(w, b->rec_w, (size_t)T * K * 4, cudaMemcpyDeviceToDevice, st));
  if (sg) CK(cudaMemcpyAsync(sg, b->rec_sg, (size_t)T * 4, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

extern "C" int moe_block_debug_set_wait(moe_block_t* b, uint32_t timeout_us, int skip_arrive) {
  if (!b) return MOE_ERR_INVALID_ARG;
  b->timeout_ns = timeout_us ? (uint64_t)timeout_us * 1000ull : 500ull * 1000 * 1000;
  b->skip_arrive = skip_arrive ? 1 : 0;
  return MOE_OK;
}

extern "C" int moe_block_debug_set_trace(moe_block_t* b, void* trace_device) {
  if (!b) return MOE_ERR_INVALID_ARG;
  b->trace = (uint64_t*)trace_device;
  return MOE_OK;
}

extern "C" int moe_block_last_launch_count(moe_block_t* b) { return b ? b->last_launches : 0; }

// ---------------------------------------------------------------- stacked decoder layers

struct moe_stack {
  moe_block_config_t cfg;
  int n_layers = 0;
  float eps = 0.f;
  moe_block** layers = nullptr;
  bool* loaded = nullptr;
  uint16_t* buf[2] = {nullptr, nullptr};   // the residual stream between layers, [max_tokens][H] fp16 each
};

extern "C" void moe_stack_destroy(moe_stack_t* s) {
  if (!s) return;
  if (s->layers)
    for (int l = 0; l < s->n_layers; ++l) moe_block_destroy(s->layers[l]);
  cudaFree(s->buf[0]);
  cudaFree(s->buf[1]);
  delete[] s->layers;
  delete[] s->loaded;
  delete s;
}

extern "C" int moe_stack_create(const moe_block_config_t* cfg, int n_layers, float eps, moe_stack_t** out) {
  if (!cfg || !out || n_layers < 1 || n_layers > 4096 || !(eps > 0.f)) return MOE_ERR_INVALID_ARG;
  {
    const int st = check_config(*cfg);
    if (st != MOE_OK) return st;
  }
  moe_stack* s = new (std::nothrow) moe_stack;
  if (!s) return MOE_ERR_CUDA;
  s->cfg = *cfg;
  s->eps = eps;
  s->layers = new (std::nothrow) moe_block*[n_layers]();
  s->loaded = new (std::nothrow) bool[n_layers]();
  if (!s->layers || !s->loaded) { moe_stack_destroy(s); return MOE_ERR_CUDA; }
  for (int l = 0; l < n_layers; ++l) {
    const int st = moe_block_create(cfg, &s->layers[l]);
    if (st != MOE_OK) { s->n_layers = l; moe_stack_destroy(s); return st; }
    s->n_layers = l + 1;
  }
  const size_t bytes = (size_t)cfg->max_tokens * cfg->hidden * 2;
  cudaError_t e = cudaMalloc(&s->buf[0], bytes);
  if (e == cudaSuccess) e = cudaMalloc(&s->buf[1], bytes);
  if (e != cudaSuccess) { moe_stack_destroy(s); return cuda_fail(e, "moe_stack_create"); }
  *out = s;
  return MOE_OK;
}

extern "C" int moe_stack_load_layer(moe_stack_t* s, int layer, const moe_block_weights_t* w, int on_device,
                                    void* stream) {
  if (!s || !w || layer < 0 || layer >= s->n_layers || !w->rms_gamma) return MOE_ERR_INVALID_ARG;
  const int st = moe_block_load_weights(s->layers[layer], w, on_device, stream);
  if (st == MOE_OK) s->loaded[layer] = true;
  return st;
}

extern "C" int moe_stack_forward(moe_stack_t* s, const void* h_in, void* h_out, int T, void* per_layer_out,
                                 void* stream) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > s->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!h_in || !h_out || !aligned16(h_in) || !aligned16(h_out)) return MOE_ERR_INVALID_ARG;
  if (per_layer_out && !aligned16(per_layer_out)) return MOE_ERR_INVALID_ARG;
  // the prompt-chunk path reads its whole input before it writes, but not within one kernel: a single layer
  // may not alias there
  if (s->n_layers == 1 && T > DEC_TMAX && h_in == h_out) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < s->n_layers; ++l)
    if (!s->loaded[l]) return MOE_ERR_NOT_LOADED;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t plane = (size_t)T * s->cfg.hidden;
  const uint16_t* in = (const uint16_t*)h_in;
  for (int l = 0; l < s->n_layers; ++l) {
    moe_block* b = s->layers[l];
    uint16_t* out = l == s->n_layers - 1 ? (uint16_t*)h_out : s->buf[l & 1];
    uint16_t* rec = per_layer_out ? (uint16_t*)per_layer_out + (size_t)l * plane : nullptr;
    // the decode kernels write the per-layer record themselves; the chunk path gets a copy
    const bool dec = T <= DEC_TMAX || !b->chunk;
    int r = run_forward(b, in, out, T, b->gamma, s->eps, st, dec ? rec : nullptr);
    if (r != MOE_OK) return r;
    if (rec && !dec) CK(cudaMemcpyAsync(rec, out, plane * 2, cudaMemcpyDeviceToDevice, st));
    in = out;
  }
  return MOE_OK;
}

extern "C" int moe_stack_get_status(moe_stack_t* s, uint32_t* flags) {
  if (!s) return MOE_ERR_INVALID_ARG;
  uint32_t all = 0;
  int result = MOE_OK;
  for (int l = 0; l < s->n_layers; ++l) {
    uint32_t f = 0;
    const int r = moe_block_get_status(s->layers[l], &f);
    all |= f;
    if (r != MOE_OK && result == MOE_OK) result = r;
  }
  if (flags) *flags = all;
  return result;
}

extern "C" moe_block_t* moe_stack_layer(moe_stack_t* s, int layer) {
  if (!s || layer < 0 || layer >= s->n_layers) return nullptr;
  return s->layers[layer];
}
