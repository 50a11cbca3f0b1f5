"""Seeded test workloads: synth draws the inputs; the oracle's exact float64 router logits decide which
tokens to redraw so that every token's k-th/(k+1)-th expert-logit gap is at least 1e-2 (the block
specification's rule for bit-exact expert ids; routing flips below a 0.015 gap are the failure mode the
TensorFold pull request #3239 reports under "Receipts")."""
import numpy as np

import oracle.moe_oracle as O
from w4a16_top_mixture_gb300 import synth

MIN_GAP = 1e-2


def gaps(logits_e, k):
    s = -np.sort(-logits_e, axis=-1)
    return s[:, k - 1] - s[:, k]


def make_case(cfg, T, seed, routing="uniform", layer=0, max_iter=64):
    w = synth.gen_layer(cfg, seed, layer)
    attempts = {}
    x = synth.gen_x(cfg, T, seed, attempts=attempts)
    for _ in range(max_iter):
        if routing == "zipf":
            w["router_q"], w["router_s"], w["router_b"] = synth.zipf_router(cfg, x, seed, layer,
                                                                             attempt=sum(attempts.values()))
        Wr = O.dequant_int8(w["router_q"], w["router_s"], w["router_b"])
        lg = x.astype(np.float64) @ Wr.T
        bad = np.nonzero(gaps(lg[:, :cfg.n_experts], cfg.top_k) < MIN_GAP)[0]
        if len(bad) == 0:
            return w, x
        for t in bad:
            attempts[int(t)] = attempts.get(int(t), 0) + 1
            x[t] = synth.gen_token(cfg, seed, int(t), attempts[int(t)])
    raise RuntimeError("could not draw a gap-respecting case")


def rel_err(out_gpu, out_ref):
    """max |err| / RMS(out_ref) over the whole output."""
    ref = np.asarray(out_ref, np.float64)
    err = np.abs(np.asarray(out_gpu, np.float64) - ref).max()
    return err / np.sqrt(np.mean(ref * ref))


def structural(out_gpu, r):
    """The block gates of the Chimera notebook (section 5 summary): cosine, norm ratio and the shared branch's
    share of the move away from the routed half."""
    g = np.asarray(out_gpu, np.float64).ravel()
    ref = r["out"].ravel()
    cos = float(g @ ref / (np.linalg.norm(g) * np.linalg.norm(ref)))
    ratio = float(np.linalg.norm(g) / np.linalg.norm(ref))
    routed = r["routed"].ravel()
    moved = np.linalg.norm(g - routed) / np.linalg.norm(ref - routed)
    return cos, ratio, moved


def half_ulp16(v):
    """Half a unit in the last place of the fp16 value nearest to v (the rounding error of a correctly rounded
    fp16 result)."""
    a = np.abs(np.asarray(v, np.float64)).astype(np.float16).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 11)


def check_tol(out_gpu, out_ref, tol=2e-3):
    """The output bound for fp16 outputs with fp32 accumulation: |err| <= tol * RMS(out_ref) on top of the
    fp16 output's own rounding (half an ulp of the reference value). The bound without that term is unreachable
    by any fp16 output once |out| reaches ~4 RMS: even the correctly rounded float64 result then misses it.
    Returns (ok, max excess over the rounding / RMS, plain max|err| / RMS)."""
    ref = np.asarray(out_ref, np.float64)
    err = np.abs(np.asarray(out_gpu, np.float64) - ref)
    rms = np.sqrt(np.mean(ref * ref))
    excess = (err - half_ulp16(ref)).clip(min=0.0).max() / rms
    return bool(excess <= tol), float(excess), float(err.max() / rms)


def quantize_acts(x, chunk=32):
    """The decode kernels' activation grid, written out: every 32-column chunk of a token is scaled by the power
    of two 2^(15 - e) (e the least integer with max|x_chunk| < 2^e), rounded to the nearest integer (ties to
    even) and clamped to +-32767, then scaled back. The kernels' integer dot products are exact on these
    values, so the oracle evaluated at quantize_acts(x) predicts the kernels' logits up to fp32 rounding."""
    x = np.asarray(x, np.float64)
    T, H = x.shape
    xc = x.reshape(T, H // chunk, chunk)
    m = np.abs(xc).max(-1, keepdims=True)
    e = np.where(m > 0, np.floor(np.log2(np.where(m > 0, m, 1.0))) + 1, -111)
    sc = 2.0 ** (15 - e)
    q = np.clip(np.rint(xc * sc), -32767, 32767)
    return (q / sc).reshape(T, H)
