"""Seeded synthetic inputs for the W4A16 routed-MoE block (weights in the canonical layout and activations).

This module only *draws* inputs. It computes nothing the block computes: no dequantisation, no GEMV, no
routing. Tests feed what it returns both to the float64 oracle and to the CUDA path; the benchmark feeds it to
the CUDA path. Every array is a pure function of (seed, layer, tensor id, attempt), drawn from a numpy
``default_rng`` seeded with that tuple, so any tensor can be regenerated on its own.

Canonical layout (what ``moe_block_load_weights`` accepts), all row-major, quantisation groups of 64 running
along the input (reduction) dimension of each output row:

  router_q    uint8 [E+1, H]      int8 codes 0..255; rows 0..E-1 are the experts, row E is the shared gate
  router_s/b  fp16  [E+1, H/64]   w = s*q + b per group
  exp_gate_q  uint8 [E, I, H/2]   int4 codes, two per byte: element 2c is the low nibble, 2c+1 the high one
  exp_gate_s/b fp16 [E, I, H/64]
  exp_up_*    same as exp_gate_*
  exp_down_q  uint8 [E, H, I/2], exp_down_s/b fp16 [E, H, I/64]
  sh_gate_q   uint8 [Is, H], sh_gate_s/b fp16 [Is, H/64]   (int8 codes)
  sh_up_*     same as sh_gate_*
  sh_down_q   uint8 [H, Is], sh_down_s/b fp16 [H, Is/64]
  rms_gamma   fp16  [H]           only for the stacked (RMSNorm + residual) configuration

Value recipe (Qwen3.6-35B-A3B decode demo, section 5: synthetic weights "in a representative range"; the
configuration list of the block under test fixes the int4 part): experts q ~ U{0..15}, s ~ U(0.005, 0.02)
rounded to fp16, b = -8 s; router and shared expert q ~ U{0..255}, s ~ U(0.005, 0.02)/16, b = -128 s (the same
weight range as the int4 experts); x ~ N(0, 1) rounded to fp16; gamma ~ U(0.9, 1.1).
"""
from __future__ import annotations

import dataclasses

import numpy as np

GROUP = 64

# tensor ids used in the seed tuple; fixed forever so stored fixtures stay valid
_TID = {
    "router": 1, "exp_gate": 2, "exp_up": 3, "exp_down": 4, "sh_gate": 5, "sh_up": 6, "sh_down": 7,
    "gamma": 8, "x": 9, "zipf_perm": 10, "zipf_gumbel": 11, "zipf_noise": 12,
}


@dataclasses.dataclass(frozen=True)
class BlockConfig:
    hidden: int = 2048
    n_experts: int = 256
    top_k: int = 8
    expert_inter: int = 512
    shared_inter: int = 512
    group: int = GROUP

    def as_dict(self):
        return dataclasses.asdict(self)


TINY = BlockConfig(hidden=512, n_experts=32, top_k=4, expert_inter=128, shared_inter=128)
PROD = BlockConfig()


def _rng(seed, layer, tid, *extra):
    return np.random.default_rng([int(seed), int(layer), int(tid), *[int(e) for e in extra]])


def _uniform_bytes(rng, shape):
    n = int(np.prod(shape))
    words = rng.bit_generator.random_raw((n + 7) // 8)
    # little-endian byte view of 64-bit draws (identical on x86_64 and aarch64)
    return words.astype("<u8", copy=False).view(np.uint8)[:n].reshape(shape)


def _scales(rng, shape, lo=0.005, hi=0.02, div=1.0):
    s = rng.uniform(lo, hi, size=shape) / div
    return s.astype(np.float16)


def int4_tensor(rng, rows_shape, in_dim):
    """Packed int4 codes uniform in 0..15 (a uniform byte holds two independent uniform nibbles), fp16
    scales U(0.005, 0.02) and bias -8*scale (exact in fp16: a power-of-two multiple)."""
    q = _uniform_bytes(rng, (*rows_shape, in_dim // 2))
    s = _scales(rng, (*rows_shape, in_dim // GROUP))
    b = (s.astype(np.float32) * np.float32(-8.0)).astype(np.float16)
    return q, s, b


def int8_tensor(rng, rows_shape, in_dim):
    """int8 affine codes uniform in 0..255, fp16 scales U(0.005, 0.02)/16 and bias -128*scale."""
    q = _uniform_bytes(rng, (*rows_shape, in_dim))
    s = _scales(rng, (*rows_shape, in_dim // GROUP), div=16.0)
    b = (s.astype(np.float32) * np.float32(-128.0)).astype(np.float16)
    return q, s, b


def gen_router(cfg: BlockConfig, seed: int, layer: int = 0, attempt: int = 0):
    rng = _rng(seed, layer, _TID["router"], attempt)
    return int8_tensor(rng, (cfg.n_experts + 1,), cfg.hidden)


def gen_layer(cfg: BlockConfig, seed: int, layer: int = 0, router_attempt: int = 0, with_gamma: bool = False):
    """All weights of one block in the canonical layout (see module docstring)."""
    H, E, I, Is = cfg.hidden, cfg.n_experts, cfg.expert_inter, cfg.shared_inter
    w = {}
    w["router_q"], w["router_s"], w["router_b"] = gen_router(cfg, seed, layer, router_attempt)
    for name, rows, ind in (("exp_gate", (E, I), H), ("exp_up", (E, I), H), ("exp_down", (E, H), I)):
        w[name + "_q"], w[name + "_s"], w[name + "_b"] = int4_tensor(_rng(seed, layer, _TID[name]), rows, ind)
    for name, rows, ind in (("sh_gate", (Is,), H), ("sh_up", (Is,), H), ("sh_down", (H,), Is)):
        w[name + "_q"], w[name + "_s"], w[name + "_b"] = int8_tensor(_rng(seed, layer, _TID[name]), rows, ind)
    if with_gamma:
        w["rms_gamma"] = _rng(seed, layer, _TID["gamma"]).uniform(0.9, 1.1, size=H).astype(np.float16)
    return w


def gen_token(cfg: BlockConfig, seed: int, t: int, attempt: int = 0, stream: int = 0):
    """One activation row x_t ~ N(0, 1) rounded to fp16, drawn from its own stream so that a single token can
    be redrawn (attempt > 0) without moving any other token."""
    rng = _rng(seed, stream, _TID["x"], t, attempt)
    return rng.standard_normal(cfg.hidden).astype(np.float16)


def gen_x(cfg: BlockConfig, T: int, seed: int, stream: int = 0, attempts=None):
    attempts = attempts or {}
    x = np.empty((T, cfg.hidden), np.float16)
    for t in range(T):
        x[t] = gen_token(cfg, seed, t, attempts.get(t, 0), stream)
    return x


def gen_x_fast(cfg: BlockConfig, T: int, seed: int, stream: int = 0):
    """Bulk draw for large benchmark batches (one stream for the whole batch; not token-addressable)."""
    rng = _rng(seed, stream, _TID["x"], 1 << 30)
    return rng.standard_normal((T, cfg.hidden)).astype(np.float16)


def quantize_int8_affine(w: np.ndarray):
    """Per-group affine int8 quantisation of a float matrix [R, C]: b = group min, s = (max-min)/255 (both
    rounded to fp16), q = clip(round((w-b)/s), 0, 255). Used only to turn a designed router into codes."""
    R, C = w.shape
    g = w.reshape(R, C // GROUP, GROUP)
    lo, hi = g.min(-1), g.max(-1)
    s = ((hi - lo) / 255.0).astype(np.float16)
    s = np.where(s == 0, np.float16(1e-3), s).astype(np.float16)
    b = lo.astype(np.float16)
    q = np.clip(np.rint((g - b.astype(np.float64)[..., None]) / s.astype(np.float64)[..., None]), 0, 255)
    return q.astype(np.uint8).reshape(R, C), s, b


def zipf_router(cfg: BlockConfig, x: np.ndarray, seed: int, layer: int = 0, s_exp: float = 1.1,
                attempt: int = 0, margin: float = 0.2, noise: float = 0.05):
    """Router rows designed so that routing of the given tokens follows Zipf(s_exp) over the experts.

    1. Expert popularity p_i proportional to rank_i^-s over a seeded permutation of the experts.
    2. Per token, target logits z_t = log p + Gumbel noise; the Gumbel top-k is a Zipf draw without
       replacement. The chosen k get `margin` added, so int8 rounding of the rows cannot reorder the k-th and
       (k+1)-th logit.
    3. Router expert rows W solve W X = Z with minimum norm, plus a seeded random component orthogonal to the
       tokens (so the rows look like ordinary weights); the shared-gate row is an ordinary random int8 row.
    4. Quantise to int8 affine g64.
    The resulting routing is checked by the caller on the exact dequantised router (the gap rule).
    """
    E, H, k = cfg.n_experts, cfg.hidden, cfg.top_k
    X = x.astype(np.float64)                          # [T, H]
    T = X.shape[0]
    perm = _rng(seed, layer, _TID["zipf_perm"]).permutation(E)
    rank = np.empty(E, np.int64)
    rank[perm] = np.arange(1, E + 1)
    logp = -s_exp * np.log(rank.astype(np.float64))
    logp -= np.log(np.exp(logp).sum())
    gum = _rng(seed, layer, _TID["zipf_gumbel"], attempt).gumbel(size=(T, E))
    Z = logp[None, :] + gum
    top = np.argsort(-Z, axis=1, kind="stable")[:, :k]
    np.put_along_axis(Z, top, np.take_along_axis(Z, top, 1) + margin, 1)
    # minimum-norm solution of W X^T = Z^T  (W: [E, H])
    W = np.linalg.lstsq(X, Z, rcond=None)[0].T        # [E, H]
    N = _rng(seed, layer, _TID["zipf_noise"], attempt).standard_normal((E, H)) * noise
    Q, _ = np.linalg.qr(X.T)                         # orthonormal basis of the tokens' span [H, T]
    N -= (N @ Q) @ Q.T
    W = W + N
    q, s, b = quantize_int8_affine(W)
    sq, ss, sb = gen_router(cfg, seed, layer, attempt)
    return (np.concatenate([q, sq[E:]], 0), np.concatenate([s, ss[E:]], 0), np.concatenate([b, sb[E:]], 0))


def layer_bytes(cfg: BlockConfig) -> int:
    """All weight + scale/bias bytes of one block (every expert)."""
    return unique_weight_bytes(cfg, cfg.n_experts)


def unique_weight_bytes(cfg: BlockConfig, n_unique_experts: int) -> int:
    """Weight + scale/bias bytes one call must read: router, shared expert and each selected expert once."""
    H, I, Is, E, G = cfg.hidden, cfg.expert_inter, cfg.shared_inter, cfg.n_experts, cfg.group
    router = (E + 1) * H + (E + 1) * (H // G) * 4
    shared = 2 * (Is * H + Is * (H // G) * 4) + (H * Is + H * (Is // G) * 4)
    expert = 2 * (I * H // 2 + I * (H // G) * 4) + (H * I // 2 + H * (I // G) * 4)
    return router + shared + n_unique_experts * expert
