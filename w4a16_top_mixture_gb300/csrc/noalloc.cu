// Allocation-free routing entry point (moe_router_topk_noalloc): the router GEMV and the softmax -> top-k ->
// renormalise step of the block, reading the router in the canonical layout, with its logits scratch in a
// fixed file-scope device array instead of memory from cudaMalloc. For callers that cannot allocate device
// memory at the point of the call: serving runtimes whose own pool allocator must account for every device
// byte, and latency-critical loops that cannot afford cudaMalloc's implicit device-wide synchronisation.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "../../include/moe_block.h"
#include "topk.cuh"

namespace {

constexpr int NA_MAX_T = 64;     // largest T one call may pass
constexpr int NA_MAX_E = 512;    // largest expert count
constexpr int NA_MAX_DEV = 64;

// Scratch for the router logits of one call, [T][E+1] fp32 (131 KB). Every GPU that loads the library holds it
// until the process exits; every call shares it.
static __device__ __align__(256) float g_na_logits[NA_MAX_T * (NA_MAX_E + 1)];

std::mutex g_na_mutex;
float* g_na_ptr[NA_MAX_DEV] = {};

// logits[t][r] = sum_c (s[r][c/64] * q[r][c] + b[r][c/64]) * x[t][c], one warp per router row
__global__ void k_na_logits(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                            const uint16_t* __restrict__ b, int H, int E, const uint16_t* __restrict__ x, int T,
                            float* __restrict__ logits) {
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (r > E) return;
  for (int t = 0; t < T; ++t) {
    float acc = 0.f;
    for (int c = lane; c < H; c += 32) {
      const int g = c / 64;
      const float sv = __half2float(__ushort_as_half(s[(size_t)r * (H / 64) + g]));
      const float bv = __half2float(__ushort_as_half(b[(size_t)r * (H / 64) + g]));
      const float w = __fmaf_rn(sv, (float)q[(size_t)r * H + c], bv);
      acc = __fmaf_rn(w, __half2float(__ushort_as_half(x[(size_t)t * H + c])), acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) logits[(size_t)t * (E + 1) + r] = acc;
  }
}

// softmax over the E expert logits -> the k largest (lower index on ties) -> renormalise; sigmoid of logit E.
// One warp per token; ids ascending, each below E whatever the logits hold. EPL: logits per lane, 32 * EPL >= E.
template <int EPL>
__global__ void k_na_topk(const float* __restrict__ logits, int E, int K, int T, int32_t* __restrict__ ids,
                          float* __restrict__ w, float* __restrict__ sg) {
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* lg = logits + (size_t)t * (E + 1);
  int sel_idx;
  float sel_val;
  moe::warp_topk_lean<EPL, false>(lg, E, K, sel_idx, sel_val);
  const float mx = __shfl_sync(0xFFFFFFFFu, sel_val, 0);
  const float ex = lane < K ? expf(sel_val - mx) : 0.f;
  float z = ex;
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  int rank = 0;
  for (int i = 0; i < K; ++i) rank += (__shfl_sync(0xFFFFFFFFu, sel_idx, i) < sel_idx) ? 1 : 0;
  if (lane < K) {
    ids[(size_t)t * K + rank] = sel_idx;
    w[(size_t)t * K + rank] = ex / z;
  }
  if (lane == 0) sg[t] = 1.0f / (1.0f + expf(-lg[E]));
}

}  // namespace

extern "C" int moe_router_topk_noalloc(const uint8_t* router_q, const uint16_t* router_s, const uint16_t* router_b,
                                       int hidden, int n_experts, int top_k, const void* x, int T, int32_t* ids,
                                       float* weights, float* sgate, void* stream) {
  if (!router_q || !router_s || !router_b || !x || !ids || !weights || !sgate) return MOE_ERR_INVALID_ARG;
  if (hidden < 64 || hidden % 64 || n_experts < 1 || n_experts > NA_MAX_E || top_k < 1 || top_k > 16 ||
      top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > NA_MAX_T) return MOE_ERR_INVALID_ARG;   // beyond the fixed scratch
  if (T == 0) return MOE_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEV) return MOE_ERR_NO_DEVICE;
  float* scratch = nullptr;
  {
    // set-up once per device, with that device current: the device address of the scratch array
    std::lock_guard<std::mutex> lk(g_na_mutex);
    if (!g_na_ptr[dev]) {
      if (cudaGetSymbolAddress((void**)&g_na_ptr[dev], g_na_logits) != cudaSuccess) {
        g_na_ptr[dev] = nullptr;
        return MOE_ERR_CUDA;
      }
    }
    scratch = g_na_ptr[dev];
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int rows = n_experts + 1;
  k_na_logits<<<(rows + 7) / 8, 256, 0, st>>>(router_q, router_s, router_b, hidden, n_experts,
                                               (const uint16_t*)x, T, scratch);
  auto* topk = n_experts <= 32 ? k_na_topk<1> : n_experts <= 64 ? k_na_topk<2> : n_experts <= 128 ? k_na_topk<4>
               : n_experts <= 256 ? k_na_topk<8> : k_na_topk<16>;
  topk<<<(T + 7) / 8, 256, 0, st>>>(scratch, n_experts, top_k, T, ids, weights, sgate);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
