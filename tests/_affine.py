"""The affine checkpoint layout for tests, written in numpy independently of the library's converter: packing
canonical codes into 32-bit little-endian code words, and the expected canonical arrays of a conversion.

Layout (moe_block.h, "affine checkpoint layout"): q[rows][in * bits / 32] uint32, input 8c + j of a 4-bit word c
in bits 4j..4j+3, input 4c + j of an 8-bit word c in bits 8j..8j+7; scales and biases [rows][in / 64] in fp16 or
bf16; w = scale * q + bias. The shared gate row arrives unquantised."""
import numpy as np


def pack_words(codes, bits):
    """codes [..., in] integers < 2**bits -> uint32 words [..., in * bits / 32] (shift-and-or, no byte views)."""
    codes = np.asarray(codes).astype(np.uint32)
    per = 32 // bits
    c = codes.reshape(*codes.shape[:-1], codes.shape[-1] // per, per)
    words = np.zeros(c.shape[:-1], np.uint32)
    for j in range(per):
        words |= c[..., j] << np.uint32(bits * j)
    return words


def unpack_int4_bytes(b):
    """canonical int4 bytes [..., in/2] -> codes [..., in] (input 2c low nibble of byte c)"""
    b = np.asarray(b, np.uint8)
    out = np.empty((*b.shape[:-1], b.shape[-1] * 2), np.uint8)
    out[..., 0::2] = b & 15
    out[..., 1::2] = b >> 4
    return out


def to_bf16(a):
    """float array -> bf16 bit patterns (round to nearest even)"""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def src_float(a, dtype):
    return bf16_to_f32(a) if dtype == "bf16" else np.asarray(a, np.uint16).view(np.float16).astype(np.float32)


def quantise_gate_row(v):
    """Expected int8 group-64 affine of the unquantised gate row v (float32 [H]): b = group min, s = (max - min)
    / 255 rounded to fp16, q = round-half-even((v - b) / s) clamped to 0..255 (all in fp32)."""
    g = v.reshape(-1, 64)
    mn, mx = g.min(axis=1), g.max(axis=1)
    s16 = ((mx - mn) / np.float32(255.0)).astype(np.float32).astype(np.float16)
    b16 = mn.astype(np.float16)
    s, b = s16.astype(np.float32), b16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, None] > 0, np.rint((g - b[:, None]) / s[:, None]), 0.0)
    q = np.clip(q, 0, 255).astype(np.uint8)
    return q.reshape(-1), s16, b16


def make_affine(cfg, seed, dtype="bf16", small_bits=8):
    """Random affine-layout weights of a block shape: experts 4-bit, router and shared expert small_bits (4 or 8),
    scales and biases in dtype, an unquantised shared gate row. Returns (aff dict for lib._affine_struct, the
    expected canonical arrays)."""
    rng = np.random.default_rng(seed)
    H, E, I, Is = cfg.hidden, cfg.n_experts, cfg.expert_inter, cfg.shared_inter

    def pairs(shape, lo, hi, bits):
        # near-centred weights, as in the synthetic workload: b = -(mid code) * s, jittered by 2 %
        s = rng.uniform(lo, hi, size=shape).astype(np.float32)
        b = -rng.uniform(0.98, 1.02, size=shape).astype(np.float32) * s * np.float32(2 ** (bits - 1))
        if dtype == "bf16":
            return to_bf16(s), to_bf16(b)
        return s.astype(np.float16).view(np.uint16), b.astype(np.float16).view(np.uint16)

    aff, exp = {"scale_dtype": dtype}, {}

    def tensor(name, rows_shape, ind, bits, int4_canonical, lo, hi):
        codes = rng.integers(0, 2 ** bits, size=(*rows_shape, ind), dtype=np.int64)
        s, b = pairs((*rows_shape, ind // 64), lo, hi, bits)
        aff[name] = (pack_words(codes, bits), s, b, bits)
        if int4_canonical:
            exp[name + "_q"] = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
        else:
            exp[name + "_q"] = codes.astype(np.uint8)
        exp[name + "_s"] = src_float(s, dtype).astype(np.float16)
        exp[name + "_b"] = src_float(b, dtype).astype(np.float16)

    tensor("router", (E,), H, small_bits, False, 0.0003, 0.0013)
    tensor("exp_gate", (E, I), H, 4, True, 0.005, 0.02)
    tensor("exp_up", (E, I), H, 4, True, 0.005, 0.02)
    tensor("exp_down", (E, H), I, 4, True, 0.005, 0.02)
    tensor("sh_gate", (Is,), H, small_bits, False, 0.0003, 0.0013)
    tensor("sh_up", (Is,), H, small_bits, False, 0.0003, 0.0013)
    tensor("sh_down", (H,), Is, small_bits, False, 0.0003, 0.0013)
    gate = rng.normal(0.0, 0.05, size=H).astype(np.float32)
    gate_src = to_bf16(gate) if dtype == "bf16" else gate.astype(np.float16).view(np.uint16)
    aff["shared_gate"] = gate_src
    gq, gs, gb = quantise_gate_row(src_float(gate_src, dtype))
    exp["router_q"] = np.concatenate([exp["router_q"], gq[None, :]])
    exp["router_s"] = np.concatenate([exp["router_s"], gs[None, :]])
    exp["router_b"] = np.concatenate([exp["router_b"], gb[None, :]])
    return aff, exp
