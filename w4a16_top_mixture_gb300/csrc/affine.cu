// Loader for the affine checkpoint layout (moe_block.h, "affine checkpoint layout"): conversion of group-64
// affine tensors with 32-bit code words into the canonical layout moe_block_load_weights takes. Host code only.
//
// Both machines this library is built for (x86-64 and Arm64) are little-endian, so the bytes of a code word are
// its inputs in order: a 4-bit word's bytes are the canonical int4 bytes (input 2c in the low nibble of byte c),
// an 8-bit word's bytes are the canonical int8 codes.
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/moe_block.h"

namespace {

static_assert(sizeof(uint32_t) == 4, "32-bit code words");

float bf16_to_float(uint16_t v) {
  const uint32_t u = (uint32_t)v << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// one scale, bias or gate value of the source dtype as a float
float src_value(uint16_t v, int dtype) {
  if (dtype == MOE_DTYPE_F16) {
    __half_raw r;
    r.x = v;
    return __half2float(__half(r));
  }
  return bf16_to_float(v);
}

// float -> fp16 bits, round to nearest even
uint16_t to_f16_bits(float f) {
  const __half_raw r = __half_raw(__float2half_rn(f));
  return r.x;
}

// A source scale or bias -> fp16 bits. fp16 input passes through; bf16 input converts exactly in fp16's normal
// range (bf16 has 8 significant bits, fp16 11). Fails on a non-finite value or one beyond fp16's range.
bool to_f16(uint16_t v, int dtype, uint16_t& out) {
  const float f = src_value(v, dtype);
  if (!std::isfinite(f)) return false;
  out = dtype == MOE_DTYPE_F16 ? v : to_f16_bits(f);
  return std::isfinite(src_value(out, MOE_DTYPE_F16));
}

bool scales_biases(const moe_affine_tensor_t& t, size_t ngroups, int dtype, uint16_t* s, uint16_t* b) {
  for (size_t i = 0; i < ngroups; ++i)
    if (!to_f16(t.scales[i], dtype, s[i]) || !to_f16(t.biases[i], dtype, b[i])) return false;
  return true;
}

// rows x in codes of bits 4 or 8 -> one canonical int8 code per byte
void codes_int8(const moe_affine_tensor_t& t, size_t rows, size_t in, uint8_t* dst) {
  if (t.bits == 8) {
    std::memcpy(dst, t.q, rows * in);
    return;
  }
  for (size_t i = 0; i < rows * in; ++i) dst[i] = (uint8_t)((t.q[i / 8] >> (4 * (i % 8))) & 15u);
}

// rows x in 4-bit codes -> canonical int4 bytes
void codes_int4(const moe_affine_tensor_t& t, size_t rows, size_t in, uint8_t* dst) {
  std::memcpy(dst, t.q, rows * in / 2);
}

bool tensor_ok(const moe_affine_tensor_t& t, bool int4_only) {
  return t.q && t.scales && t.biases && (t.bits == 4 || (!int4_only && t.bits == 8));
}

}  // namespace

extern "C" void moe_affine_free(moe_block_weights_t* w) {
  if (!w) return;
  // every converted array lives in one allocation that starts at router_q
  delete[] const_cast<uint8_t*>(w->router_q);
  std::memset(w, 0, sizeof(*w));
}

extern "C" int moe_affine_convert(const moe_block_config_t* cfg, const moe_affine_weights_t* src,
                                  moe_block_weights_t* out) {
  if (!cfg || !src || !out) return MOE_ERR_INVALID_ARG;
  const size_t H = cfg->hidden, E = cfg->n_experts, I = cfg->expert_inter, Is = cfg->shared_inter;
  if (cfg->group_size != 64 || H < 64 || H % 64 || I < 64 || I % 64 || Is < 64 || Is % 64 || cfg->n_experts < 1)
    return MOE_ERR_INVALID_ARG;
  if (src->scale_dtype != MOE_DTYPE_F16 && src->scale_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (!tensor_ok(src->router, false) || !tensor_ok(src->exp_gate, true) || !tensor_ok(src->exp_up, true) ||
      !tensor_ok(src->exp_down, true) || !tensor_ok(src->sh_gate, false) || !tensor_ok(src->sh_up, false) ||
      !tensor_ok(src->sh_down, false) || !src->shared_gate)
    return MOE_ERR_INVALID_ARG;
  const int dt = src->scale_dtype;

  // one allocation: codes first (router first, so that moe_affine_free finds the base), then the fp16 pairs
  const size_t n_rq = (E + 1) * H, n_egq = E * I * H / 2, n_edq = E * H * I / 2, n_sq = Is * H;
  const size_t n_rs = (E + 1) * (H / 64), n_egs = E * I * (H / 64), n_eds = E * H * (I / 64), n_ss = Is * (H / 64);
  const size_t code_bytes = n_rq + 2 * n_egq + n_edq + 3 * n_sq;
  const size_t pair_elems = n_rs + 2 * n_egs + n_eds + 3 * n_ss;
  uint8_t* base = new (std::nothrow) uint8_t[code_bytes + 4 * pair_elems + 16];
  if (!base) return MOE_ERR_INVALID_ARG;
  uint8_t* cp = base;
  auto codes = [&](size_t n) { uint8_t* r = cp; cp += n; return r; };
  uint16_t* sp = reinterpret_cast<uint16_t*>(base + ((code_bytes + 15) & ~(size_t)15));
  auto halves = [&](size_t n) { uint16_t* r = sp; sp += n; return r; };
  uint8_t *rq = codes(n_rq), *egq = codes(n_egq), *euq = codes(n_egq), *edq = codes(n_edq);
  uint8_t *sgq = codes(n_sq), *suq = codes(n_sq), *sdq = codes(n_sq);
  uint16_t *rs = halves(n_rs), *rb = halves(n_rs);
  uint16_t *egs = halves(n_egs), *egb = halves(n_egs), *eus = halves(n_egs), *eub = halves(n_egs);
  uint16_t *eds = halves(n_eds), *edb = halves(n_eds);
  uint16_t *sgs = halves(n_ss), *sgb = halves(n_ss), *sus = halves(n_ss), *sub = halves(n_ss);
  uint16_t *sds = halves(n_ss), *sdb = halves(n_ss);

  bool ok = true;
  // router rows 0..E-1, then the shared gate row E quantised here
  codes_int8(src->router, E, H, rq);
  ok = ok && scales_biases(src->router, E * (H / 64), dt, rs, rb);
  for (size_t g = 0; ok && g < H / 64; ++g) {
    float v[64], mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < 64; ++i) {
      v[i] = src_value(src->shared_gate[g * 64 + i], dt);
      if (!std::isfinite(v[i])) ok = false;
      mn = std::fmin(mn, v[i]);
      mx = std::fmax(mx, v[i]);
    }
    const uint16_t s16 = to_f16_bits((mx - mn) / 255.0f), b16 = to_f16_bits(mn);
    const float s = src_value(s16, MOE_DTYPE_F16), b = src_value(b16, MOE_DTYPE_F16);
    rs[E * (H / 64) + g] = s16;
    rb[E * (H / 64) + g] = b16;
    for (int i = 0; i < 64; ++i) {
      const long q = s > 0.f ? std::lrint((v[i] - b) / s) : 0;
      rq[E * H + g * 64 + i] = (uint8_t)(q < 0 ? 0 : q > 255 ? 255 : q);
    }
  }
  codes_int4(src->exp_gate, E * I, H, egq);
  codes_int4(src->exp_up, E * I, H, euq);
  codes_int4(src->exp_down, E * H, I, edq);
  ok = ok && scales_biases(src->exp_gate, n_egs, dt, egs, egb) && scales_biases(src->exp_up, n_egs, dt, eus, eub) &&
       scales_biases(src->exp_down, n_eds, dt, eds, edb);
  codes_int8(src->sh_gate, Is, H, sgq);
  codes_int8(src->sh_up, Is, H, suq);
  codes_int8(src->sh_down, H, Is, sdq);
  ok = ok && scales_biases(src->sh_gate, n_ss, dt, sgs, sgb) && scales_biases(src->sh_up, n_ss, dt, sus, sub) &&
       scales_biases(src->sh_down, n_ss, dt, sds, sdb);
  if (!ok) {
    delete[] base;
    return MOE_ERR_INVALID_ARG;
  }
  moe_block_weights_t w;
  w.router_q = rq; w.router_s = rs; w.router_b = rb;
  w.exp_gate_q = egq; w.exp_gate_s = egs; w.exp_gate_b = egb;
  w.exp_up_q = euq; w.exp_up_s = eus; w.exp_up_b = eub;
  w.exp_down_q = edq; w.exp_down_s = eds; w.exp_down_b = edb;
  w.sh_gate_q = sgq; w.sh_gate_s = sgs; w.sh_gate_b = sgb;
  w.sh_up_q = suq; w.sh_up_s = sus; w.sh_up_b = sub;
  w.sh_down_q = sdq; w.sh_down_s = sds; w.sh_down_b = sdb;
  w.rms_gamma = src->rms_gamma;
  *out = w;
  return MOE_OK;
}
