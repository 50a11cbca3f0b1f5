/*
 * moe_block.h -- C ABI of the GB300 (sm_103a) W4A16 routed Mixture-of-Experts FFN block.
 *
 * The operation (Qwen3.6-35B-A3B decode demo on the Chimera GPNPU, section 5 "Validate the MoE FFN block",
 * and TensorFold pull request #3239, section "Design"):
 *
 *   logits = W_R x               W_R: int8 group-64 affine, E expert rows stacked with the shared-gate row
 *   p      = softmax(logits[0:E]);  S = top_k(p);  w_j = p_j / sum_{i in S} p_i        (section 5.2 ordering)
 *   y_j    = Wd_j (silu(Wg_j x) * (Wu_j x))            routed experts, int4 group-64 affine (SwiGLU)
 *   ys     = Wsd  (silu(Wsg x) * (Wsu x))              shared expert, int8 group-64 affine
 *   out    = sum_{j in S} w_j y_j + sigmoid(logits[E]) * ys
 *
 * Activations are fp16 ("W4A16": weights int4/int8, activations fp16); every product is accumulated in fp32
 * and the output is rounded to fp16 once. Dequantisation is w = s * q + b per group of 64 inputs, with
 * unsigned codes and fp16 s, b.
 *
 * Canonical weight layout accepted by moe_block_load_weights (row-major, groups of 64 along each output row's
 * input dimension; int4 codes two per byte, element 2c in the low nibble of byte c, element 2c+1 in the high):
 *   router_q  [E+1][H] u8,  router_s/b  [E+1][H/64] fp16    row E is the shared-expert gate
 *   exp_gate_q[E][I][H/2] u8, exp_gate_s/b [E][I][H/64] fp16  (exp_up_* alike)
 *   exp_down_q[E][H][I/2] u8, exp_down_s/b [E][H][I/64] fp16
 *   sh_gate_q [Is][H] u8,   sh_gate_s/b [Is][H/64] fp16      (sh_up_* alike)
 *   sh_down_q [H][Is] u8,   sh_down_s/b [H][Is/64] fp16
 *   rms_gamma [H] fp16 (stacked blocks only; NULL otherwise)
 * fp16 values are passed as their 16-bit patterns (uint16_t).
 *
 * Conventions. Every entry point returns an int status (MOE_OK = 0, negative on error) and validates its
 * arguments before touching any state; nothing throws or aborts across the ABI. Streams are cudaStream_t
 * values passed as void* (NULL = legacy default stream). Calls on one handle must not overlap in time.
 */
#ifndef MOE_BLOCK_H
#define MOE_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,     /* null / misaligned pointer, T out of range, bad index */
  MOE_ERR_UNSUPPORTED = -2,     /* configuration has no kernel (see moe_block_create) */
  MOE_ERR_NOT_LOADED = -3,      /* forward before load_weights */
  MOE_ERR_CUDA = -4,            /* a CUDA runtime call failed; moe_last_cuda_error() names it */
  MOE_ERR_DEVICE_TIMEOUT = -5,  /* a bounded device-side wait ran out (see moe_block_get_status) */
  MOE_ERR_NO_DEVICE = -6,       /* no sm_103 device current */
};

typedef struct moe_block moe_block_t;   /* opaque, owned by the library */

typedef struct {
  int hidden;        /* H: 512, 1024 or 2048 */
  int n_experts;     /* E: 1..512 */
  int top_k;         /* k: 1..min(E, 16) */
  int expert_inter;  /* I: multiple of 64, 64..1024 */
  int shared_inter;  /* Is: multiple of 64, 64..1024 */
  int group_size;    /* must be 64 */
  int max_tokens;    /* largest T any forward will pass: 1..4096 (sizes the scratch allocated at create) */
} moe_block_config_t;

typedef struct {
  const uint8_t *router_q;   const uint16_t *router_s,   *router_b;
  const uint8_t *exp_gate_q; const uint16_t *exp_gate_s, *exp_gate_b;
  const uint8_t *exp_up_q;   const uint16_t *exp_up_s,   *exp_up_b;
  const uint8_t *exp_down_q; const uint16_t *exp_down_s, *exp_down_b;
  const uint8_t *sh_gate_q;  const uint16_t *sh_gate_s,  *sh_gate_b;
  const uint8_t *sh_up_q;    const uint16_t *sh_up_s,    *sh_up_b;
  const uint8_t *sh_down_q;  const uint16_t *sh_down_s,  *sh_down_b;
  const uint16_t *rms_gamma; /* may be NULL */
} moe_block_weights_t;

/* ---- affine checkpoint layout (TensorFold #3239, "Receipts": the block run from the published 4-bit affine
 * checkpoint of Qwen3.6-35B-A3B). The pages name that checkpoint but give no layout; this loader reads the
 * plainest one for group-64 affine tensors:
 *   q       [rows][in * bits / 32] uint32 words along the input dimension, little-endian: with bits = 4 word c
 *           holds inputs 8c..8c+7, input 8c + j in bits 4j..4j+3; with bits = 8 word c holds inputs 4c..4c+3,
 *           input 4c + j in bits 8j..8j+7. Batched matrices (the experts) follow one another.
 *   scales  [rows][in/64], biases [rows][in/64], fp16 or bf16 (scale_dtype): w = scales * q + biases.
 * Read as bytes, a 4-bit word is the canonical int4 row (element 2c in the low nibble of byte c); 4-bit router
 * and shared-expert tensors widen to the canonical int8 codes exactly, and bf16 scales and biases convert to fp16
 * exactly in fp16's normal range. The shared expert's gate row (row E of the canonical router) comes
 * unquantised and is quantised here to int8 group-64 affine: b = group min, s = (max - min) / 255 rounded to
 * fp16, q = round((w - b) / s) clamped to 0..255. All pointers are host memory. */
enum { MOE_DTYPE_F16 = 0, MOE_DTYPE_BF16 = 1 };

typedef struct {
  const uint32_t *q;
  const uint16_t *scales, *biases;
  int bits;   /* 4 or 8; the routed experts' tensors must be 4 */
} moe_affine_tensor_t;

typedef struct {
  moe_affine_tensor_t router;                 /* [E][H] */
  moe_affine_tensor_t exp_gate, exp_up;       /* [E][I][H] */
  moe_affine_tensor_t exp_down;               /* [E][H][I] */
  moe_affine_tensor_t sh_gate, sh_up;         /* [Is][H] */
  moe_affine_tensor_t sh_down;                /* [H][Is] */
  const uint16_t *shared_gate;                /* [H], scale_dtype */
  const uint16_t *rms_gamma;                  /* [H] fp16, or NULL */
  int scale_dtype;                            /* MOE_DTYPE_F16 or MOE_DTYPE_BF16 */
} moe_affine_weights_t;

/* Convert affine-layout weights into the canonical layout, in host buffers the library allocates: *out then
 * points at them (rms_gamma at the caller's). Free them with moe_affine_free. Host work only: no device is
 * touched. MOE_ERR_INVALID_ARG: a NULL pointer, bits other than 4 / 8 (4 for the routed experts), an unknown
 * scale_dtype, a value that is not finite or overflows fp16, or host memory that cannot be allocated. */
MOE_API int moe_affine_convert(const moe_block_config_t *cfg, const moe_affine_weights_t *src,
                               moe_block_weights_t *out);
MOE_API void moe_affine_free(moe_block_weights_t *w);

/* moe_affine_convert + moe_block_load_weights (from host memory) + moe_affine_free. */
MOE_API int moe_block_load_affine(moe_block_t *blk, const moe_affine_weights_t *src, void *stream);

/* Create a handle for one block on the current CUDA device. Allocates the device weight store (repacked
 * layout) and all scratch for max_tokens, so forward never allocates. Refuses configurations it has no
 * kernel for with MOE_ERR_UNSUPPORTED. *out is set only on success. */
MOE_API int moe_block_create(const moe_block_config_t *cfg, moe_block_t **out);

/* Copy and repack the canonical weights into the handle. weights_on_device = 1: the pointers are device
 * memory; 0: host memory (copied through a temporary device buffer). The caller keeps ownership and may free
 * its buffers once this returns (the call synchronises `stream`). A handle that serves prompt chunks
 * (max_tokens > 16) forms s * q in fp16 (as an exact pair of halves) on its chunk path, so it refuses with
 * MOE_ERR_INVALID_ARG, and stays unloaded, when a scale is not finite or |s| * (largest code: 15 for int4, 255
 * for int8) reaches 65504; decode-only handles compute in fp32 and have no such limit. */
MOE_API int moe_block_load_weights(moe_block_t *blk, const moe_block_weights_t *w, int weights_on_device, void *stream);

/* out[T][H] = block(x[T][H]). x and out are caller-owned device buffers of fp16, 16-byte aligned, not
 * aliasing. 0 <= T <= max_tokens (T = 0 is a no-op). Asynchronous on `stream`, no host synchronisation and no
 * allocation, so it can be captured in a CUDA graph. T <= 16 runs a fused decode kernel; larger T the
 * prompt-chunk path.
 *
 * Residency. The decode kernels (one launch of one CTA per SM) hand results between their CTAs through
 * grid-wide counts, so all CTAs of a launch must be resident at once; moe_block_create checks that the grid
 * fits the device. A kernel of another stream, process or client that holds SMs while a forward runs can keep
 * some of its CTAs from starting: the others then wait, bounded (500 ms by default), and the call ends without
 * its result, which moe_block_get_status (and moe_block_forward_host, which reads the status itself) reports
 * as MOE_ERR_DEVICE_TIMEOUT. Run forward with the SMs to itself, or poll the status.
 *
 * After such an error the handle's single-token (T = 1) kernel computes nothing, and leaves out unwritten, until
 * moe_block_get_status has reported the error and reset the handle: its grid-wide counts and published routing
 * words are consistent again only then. The refused call adds bit 128 to the status flags. */
MOE_API int moe_block_forward(moe_block_t *blk, const void *x, void *out, int T, void *stream);

/* Same computation with HOST buffers: copies x to the device, runs forward and copies out back, then
 * synchronises `stream`. x_host/out_host should be pinned for full copy speed. */
MOE_API int moe_block_forward_host(moe_block_t *blk, const void *x_host, void *out_host, int T, void *stream);

/* Stacked configuration: h_out = h_in + block(RMSNorm(h_in)) with RMSNorm y = h / sqrt(mean(h^2) + eps) *
 * gamma (notebook section 7: the decoder layer wraps the MoE op in RMSNorm and a residual add). Needs
 * rms_gamma loaded. h_in and h_out fp16 device [T][H]; they may alias. */
MOE_API int moe_block_forward_residual(moe_block_t *blk, const void *h_in, void *h_out, int T, float eps, void *stream);

/* Waits for the stream of the handle's last forward call (that stream must still exist; work replayed from a
 * CUDA graph on another stream must be synchronised by the caller first), then returns MOE_OK, or
 * MOE_ERR_DEVICE_TIMEOUT if a bounded device-side wait ran out in any earlier call (the handle's device state
 * is then reset, so the next call starts clean). *flags (may be NULL) receives the raw device error bits: 1 the
 * router logits, 2 the shared-expert h, 4 the routed h, 8 a weight copy, 16 a shared-memory region, 32 the
 * routing plan were not ready in time; 128 a single-token call found an earlier error not yet reset and computed
 * nothing; 512 a prompt-chunk GEMM wait ran out. */
MOE_API int moe_block_get_status(moe_block_t *blk, uint32_t *flags);

/* ---- stacked decoder layers (notebook section 7: the decoder layer wraps the MoE block in RMSNorm and a
 * residual add; TensorFold #3239, "What this changes": staged references compare each layer's local error
 * with the error chained through the stack) ----
 *
 * A stack holds n_layers blocks of one shape, each with its own weights and RMSNorm gamma, and runs
 *   h_{l+1} = h_l + block_l(RMSNorm_l(h_l)),  l = 0 .. n_layers-1,   RMSNorm(h) = h / sqrt(mean(h^2) + eps) * gamma
 * on fp16 hidden states: h_in = h_0, h_out = h_{n_layers}; between layers the residual stream is fp16. */
typedef struct moe_stack moe_stack_t;   /* opaque, owned by the library */

/* n_layers >= 1 blocks of shape *cfg (every layer allocates its own weight store and scratch, as
 * moe_block_create does), plus two [max_tokens][H] fp16 buffers for the residual stream. eps > 0. */
MOE_API int moe_stack_create(const moe_block_config_t *cfg, int n_layers, float eps, moe_stack_t **out);

/* Weights of layer `layer` (0-based) in the canonical layout of moe_block_load_weights; rms_gamma is
 * required. Synchronises `stream`; the caller may free its buffers on return. */
MOE_API int moe_stack_load_layer(moe_stack_t *stk, int layer, const moe_block_weights_t *w, int weights_on_device,
                                 void *stream);

/* h_out[T][H] = the stack applied to h_in[T][H] (fp16 device buffers, 16-byte aligned; h_out may alias h_in
 * when T <= 16 or n_layers > 1). per_layer_out: NULL, or fp16 device [n_layers][T][H] that receives h_{l+1}
 * for every layer l (the per-layer record of the staged-reference method). Every layer must be loaded. The
 * layers are issued back to back on `stream` as programmatic-dependent launches (at T = 1 the next layer's CTAs
 * become resident and load their weight-only rows while the current layer runs); no host synchronisation and
 * no allocation. */
MOE_API int moe_stack_forward(moe_stack_t *stk, const void *h_in, void *h_out, int T, void *per_layer_out,
                              void *stream);

/* moe_block_get_status over every layer (flags: the OR of their error bits). */
MOE_API int moe_stack_get_status(moe_stack_t *stk, uint32_t *flags);

/* The handle of layer `layer` (owned by the stack; for the per-block test hooks), or NULL. */
MOE_API moe_block_t *moe_stack_layer(moe_stack_t *stk, int layer);

MOE_API void moe_stack_destroy(moe_stack_t *stk);

MOE_API void moe_block_destroy(moe_block_t *blk);
MOE_API const char *moe_block_strerror(int status);
MOE_API const char *moe_last_cuda_error(void);

/* ---- test hooks (not on the hot path) ---- */

/* Dequantised fp32 matrix from the handle's repacked store, written to out_device (device, row-major in the
 * canonical orientation). which: 0 router [E+1][H], 1 exp gate [I][H], 2 exp up [I][H], 3 exp down [H][I],
 * 4 shared gate [Is][H], 5 shared up [Is][H], 6 shared down [H][Is]; index = expert for 1..3. */
MOE_API int moe_block_debug_dequant(moe_block_t *blk, int which, int index, float *out_device, void *stream);

/* Routing of the last forward call, copied to device buffers (any may be NULL): ids [T][k] int32 ascending,
 * weights [T][k] fp32 aligned with ids, sigmoid gate [T] fp32 for its first T tokens; logits [T][E+1] fp32 only
 * for calls with T <= 16 (must be NULL otherwise). */
MOE_API int moe_block_debug_last_routing(moe_block_t *blk, int T, float *logits, int32_t *ids, float *weights,
                                 float *sgate, void *stream);

/* Test control of the bounded device waits: timeout_us = microseconds any device-side wait may last before
 * it gives up (0 = the default, 500 ms); skip_arrive = 1 withholds one arrival in the next forward call only:
 * in the decode kernels the logits count of the CTA holding router row 0 (single token) or of CTA 0 (more
 * tokens), so every CTA's bounded wait for the logits runs out; on the prompt-chunk path CTA 0's first weight
 * copy of the router GEMM, so that CTA's waits for it run out. The call ends early with an error bit set and
 * wrong outputs, and the host sees MOE_ERR_DEVICE_TIMEOUT from moe_block_get_status. No fault is involved. */
MOE_API int moe_block_debug_set_wait(moe_block_t *blk, uint32_t timeout_us, int skip_arrive);

/* Phase timestamps for performance analysis: when trace_device is non-NULL, every later decode call writes
 * SM clock stamps (clock64) at its phase boundaries into trace_device[cta * 32 + slot], %globaltimer
 * nanoseconds at the CTA's start and end into slots 30 and 31 (to place every CTA on one time axis), and
 * per-warp clock stamps into trace_device[32 * G + (cta * 16 + warp) * 4 + k] (G = number of SMs). A slot a
 * call does not reach holds 0. A chunk call (T > 16) writes instead the stamps of CTA 0's first 64 K-tiles
 * of its expert gate/up GEMM launch into trace_device[event * 64 + k], events 0..6: copies issued,
 * dequantisation start and end, MMAs issued, fold start and end, A seen ready by the MMA issuer. trace_device
 * is uint64 device memory of at least 96 * number-of-SMs entries, caller-owned; NULL switches tracing off. */
MOE_API int moe_block_debug_set_trace(moe_block_t *blk, void *trace_device);

/* ---- allocation-free routing ----
 * No counterpart on the pages. For callers that cannot allocate device memory at the point of the call: a
 * serving runtime whose own pool allocator must account for every device byte (memory taken with cudaMalloc
 * behind its back breaks its budget), or a latency-critical decode loop that cannot afford cudaMalloc's
 * implicit device-wide synchronisation. Computes the routing step of the block -- router logits from the CANONICAL int8 router
 * (router_q [E+1][H], router_s/b [E+1][H/64] fp16 bits, device memory), softmax over the E expert logits,
 * top-k, renormalisation, sigmoid of the shared-gate logit -- for x [T][H] fp16 (device) into ids [T][k] int32
 * (ascending), weights [T][k] fp32 and sgate [T] fp32 (device). It allocates nothing: the logits live in a
 * fixed 131 KB device array inside the library (T <= 64 tokens, E <= 512 experts; larger T or E return
 * MOE_ERR_INVALID_ARG). Every call shares that array, so calls that overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller. The first call on a device looks up the array's device
 * address once; make that first call before any stream capture. Asynchronous on `stream`. */
MOE_API int moe_router_topk_noalloc(const uint8_t *router_q, const uint16_t *router_s, const uint16_t *router_b,
                                    int hidden, int n_experts, int top_k, const void *x, int T, int32_t *ids,
                                    float *weights, float *sgate, void *stream);

/* Number of CUDA kernel launches the last forward call made. */
MOE_API int moe_block_last_launch_count(moe_block_t *blk);

/* Host-only planning query (no device, no allocation): the launch plan the fused decode kernel uses for a call
 * of T tokens on a device with num_sms SMs and max_smem bytes of opt-in shared memory per block. On MOE_OK,
 * out[0..4] = grid (CTAs), dynamic shared memory bytes, ring stages, bytes per stage, and h vectors staged in
 * shared memory. MOE_ERR_UNSUPPORTED: the shape or T has no decode plan (T > 16 uses the chunk path);
 * MOE_ERR_INVALID_ARG: a NULL pointer or a non-positive size. */
MOE_API int moe_debug_decode_plan(const moe_block_config_t *cfg, int T, int num_sms, int max_smem, int32_t *out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_BLOCK_H */
