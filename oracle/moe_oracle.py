"""Plain float64 reference of the decode-time routed MoE FFN block of Qwen3.6-35B-A3B.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA path never imports or calls this.

Sources. "Qwen3.6-35B-A3B Decode on Chimera GPNPU" (Quadric SDK notebook), section 5 "Validate the MoE FFN
block": the block computes out = routed + sigmoid(x . W_sg) * shared, the routed half being the top-k experts
and the shared half a dense SwiGLU expert; section 5.2: the router orders softmax -> top-k -> renormalise,
experts are SwiGLU, the output gate is a sigmoid. Section "Pipeline" and the key takeaways: routed experts int4,
shared expert int8, activations fp16; hidden 2048, 256 experts, top-8, shared intermediate 512. The TensorFold
pull request #3239 ("qwen27: Qwen3.6-35B-A3B on Metal on the routed path"), section "Design": 256 experts of
512 and a shared expert of 512 over a hidden width of 2048; the router runs on stored 8-bit group-64 rows
stacked with the shared gate. Section 7 of the notebook: the decoder layer wraps the MoE op in RMSNorm and a
residual add.

Readings where the pages are silent (each one is listed with its reason in the design notes):
  * affine group-64 dequantisation w = s*q + b, codes unsigned, s and b fp16;
  * int4 packing: element 2c is the low nibble of byte c, element 2c+1 the high nibble;
  * router rows 0..E-1 are the experts, row E is the shared gate; the softmax runs over the E expert logits;
  * top-k picks the k largest logits, the lower index winning an exact tie;
  * RMSNorm y = x / sqrt(mean(x^2) + eps) * gamma (plain gamma), eps = 1e-6.

Everything is float64 and written step by step in the pages' order; numpy matmul is the only library routine
used as a step.
"""
from __future__ import annotations

import numpy as np

GROUP = 64

__all__ = [
    "unpack_int4", "dequant", "dequant_int4", "dequant_int8", "softmax", "route", "silu", "sigmoid",
    "swiglu_expert", "block_forward", "rmsnorm", "stack_forward", "Dequantizer",
]


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Codes [..., 2C] from packed bytes [..., C]: element 2c = low nibble of byte c, 2c+1 = high nibble."""
    p = packed.astype(np.int64)
    out = np.empty((*packed.shape[:-1], 2 * packed.shape[-1]), np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant(codes: np.ndarray, s: np.ndarray, b: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Affine group dequantisation W[r, c] = s[r, c // group] * q[r, c] + b[r, c // group], in float64.

    Exact: s and b are fp16 and q has at most 8 bits, so every product and sum fits in 53 bits."""
    q = codes.astype(np.float64)
    sf = np.repeat(s.astype(np.float64), group, axis=-1)
    bf = np.repeat(b.astype(np.float64), group, axis=-1)
    return sf * q + bf


def dequant_int4(packed, s, b, group: int = GROUP):
    return dequant(unpack_int4(packed), s, b, group)


def dequant_int8(q, s, b, group: int = GROUP):
    return dequant(q, s, b, group)


def softmax(v: np.ndarray) -> np.ndarray:
    m = v.max(axis=-1, keepdims=True)
    e = np.exp(v - m)
    return e / e.sum(axis=-1, keepdims=True)


def sigmoid(z):
    with np.errstate(over="ignore"):          # exp(-z) -> inf for z << 0 gives the correct limit 0
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def route(expert_logits: np.ndarray, k: int):
    """Softmax over the experts -> the k largest -> renormalise to sum 1.

    Returns ids [T, k] (ascending), weights [T, k] (aligned with ids) and the full probabilities [T, E]."""
    p = softmax(expert_logits)
    order = np.argsort(-expert_logits, axis=-1, kind="stable")[:, :k]   # largest first, lower index on ties
    ids = np.sort(order, axis=-1)
    sel = np.take_along_axis(p, ids, axis=-1)
    w = sel / sel.sum(axis=-1, keepdims=True)
    return ids, w, p


def swiglu_expert(Wg, Wu, Wd, x):
    """y = Wd (silu(Wg x) * (Wu x)) for x [T, H]; returns (y [T, H_out], h [T, I])."""
    a = x @ Wg.T
    u = x @ Wu.T
    h = silu(a) * u
    return h @ Wd.T, h


class Dequantizer:
    """Float64 views of one block's canonical weights, dequantised lazily (only the experts a call selects)."""

    def __init__(self, w: dict, group: int = GROUP):
        self.w, self.g = w, group
        self._cache = {}

    def router(self):
        if "router" not in self._cache:
            w = self.w
            self._cache["router"] = dequant_int8(w["router_q"], w["router_s"], w["router_b"], self.g)
        return self._cache["router"]

    def shared(self):
        if "shared" not in self._cache:
            w, g = self.w, self.g
            self._cache["shared"] = tuple(dequant_int8(w[n + "_q"], w[n + "_s"], w[n + "_b"], g)
                                          for n in ("sh_gate", "sh_up", "sh_down"))
        return self._cache["shared"]

    def expert(self, e: int):
        key = ("e", int(e))
        if key not in self._cache:
            w, g = self.w, self.g
            self._cache[key] = tuple(dequant_int4(w[n + "_q"][e], w[n + "_s"][e], w[n + "_b"][e], g)
                                     for n in ("exp_gate", "exp_up", "exp_down"))
        return self._cache[key]


def block_forward(w: dict, x: np.ndarray, top_k: int, group: int = GROUP, deq: Dequantizer | None = None):
    """The MoE block on tokens x [T, H] (any float dtype; taken exactly as float64).

    1. router: logits = W_R x over E+1 rows; row E is the shared gate g.
    2. routing: softmax over the E expert logits, top-k, renormalise.
    3. each selected expert: SwiGLU MLP y_j.
    4. shared expert: SwiGLU MLP ys.
    5. out = sum_j w_j y_j + sigmoid(g) ys.
    Returns a dict with every intermediate the tests compare."""
    deq = deq or Dequantizer(w, group)
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = w["router_q"].shape[0] - 1
    logits = x @ deq.router().T                       # [T, E+1]
    ids, wts, probs = route(logits[:, :E], top_k)
    g = logits[:, E]
    sg = sigmoid(g)
    Wsg, Wsu, Wsd = deq.shared()
    ys, hs = swiglu_expert(Wsg, Wsu, Wsd, x)
    H_out = Wsd.shape[0]
    routed = np.zeros((T, H_out))
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        Wg, Wu, Wd = deq.expert(e)
        y, _ = swiglu_expert(Wg, Wu, Wd, x[rows])
        routed[rows] += wts[rows, slots][:, None] * y
    out = routed + sg[:, None] * ys
    return {"out": out, "logits": logits, "ids": ids, "w": wts, "probs": probs, "sg": sg, "g": g,
            "routed": routed, "shared": ys, "hs": hs}


def rmsnorm(h: np.ndarray, gamma: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """y = h / sqrt(mean(h^2) + eps) * gamma, per row, float64 (decoder-layer RMSNorm, notebook section 7)."""
    h = np.asarray(h, np.float64)
    r = 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    return h * r * np.asarray(gamma, np.float64)


def stack_forward(layers: list, h0: np.ndarray, top_k: int, eps: float = 1e-6, group: int = GROUP):
    """h_{l+1} = h_l + block_l(RMSNorm_l(h_l)) through every layer, float64 throughout.

    Returns (h_final, per-layer dicts of block_forward plus the layer input)."""
    h = np.asarray(h0, np.float64)
    recs = []
    for w in layers:
        xn = rmsnorm(h, w["rms_gamma"], eps)
        r = block_forward(w, xn, top_k, group)
        r["h_in"], r["x_norm"] = h, xn
        h = h + r["out"]
        recs.append(r)
    return h, recs
