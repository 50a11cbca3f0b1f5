"""Stacked decoder layers through the stack entry points (moe_stack_create / moe_stack_load_layer /
moe_stack_forward): h_{l+1} = h_l + block_l(RMSNorm_l(h_l)) with eps = 1e-6 (the decoder-layer assembly of the
Chimera notebook, section 7), all layers issued by one moe_stack_forward call.

Local error per layer (the staged-reference method of TensorFold PR #3239, "Staged references": every stage fed
the engine's own input): the per-layer record of the call (per_layer_out) gives the GPU's input h_l of every
layer; the oracle forms the block input as the layer does (RMSNorm, rounded to the fp16 activation) and predicts
h_l + block(...); the GPU's h_{l+1} must agree within 2e-3 * RMS(block output) plus half an fp16 ulp of h_{l+1}
(the residual stream is fp16 between blocks). The chained error against a float64 chain from the same h_0 grows
with depth and is reported, not gated."""
import numpy as np
import pytest

import oracle.moe_oracle as O
from tests._cases import MIN_GAP, gaps, half_ulp16
from w4a16_top_mixture_gb300 import build, lib, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 2e-3
EPS = 1e-6


def _block_input(h, gamma):
    """The block's activation as the stacked layer forms it: RMSNorm of the fp16 residual, rounded to fp16
    (activations are fp16 in W4A16)."""
    return O.rmsnorm(h, gamma, EPS).astype(np.float16).astype(np.float64)


def _layers_and_input(cfg, seed, n_layers, T=1):
    """Layers whose routers respect the gap rule on the inputs of a chain rounded like the block's own
    activations (fp16 residual, fp16 block input): the GPU's layer inputs differ from it only by last-place
    roundings, far inside the 1e-2 gap."""
    h = synth.gen_x(cfg, T, seed).astype(np.float64)
    h0 = h.astype(np.float16)
    layers = []
    for l in range(n_layers):
        w = synth.gen_layer(cfg, seed, l, with_gamma=True)
        xn = _block_input(h, w["rms_gamma"])
        for attempt in range(1, 64):
            lg = xn @ O.dequant_int8(w["router_q"], w["router_s"], w["router_b"]).T
            if gaps(lg[:, :cfg.n_experts], cfg.top_k).min() >= MIN_GAP:
                break
            w["router_q"], w["router_s"], w["router_b"] = synth.gen_router(cfg, seed, l, attempt)
        layers.append(w)
        h = (h + O.block_forward(w, xn, cfg.top_k)["out"]).astype(np.float16).astype(np.float64)
    h_chain, _ = O.stack_forward(layers, h0.astype(np.float64), cfg.top_k, EPS)
    return layers, h0, h_chain


def _run_stack(cfg, layers, h0, max_tokens):
    import torch
    T = h0.shape[0]
    stk = lib.MoeStack(cfg, len(layers), max_tokens=max_tokens, eps=EPS)
    for l, w in enumerate(layers):
        stk.load_layer(l, w)
    h_in = torch.from_numpy(h0.view(np.int16)).cuda().view(torch.float16)
    rec = torch.empty((len(layers), T, cfg.hidden), dtype=torch.float16, device="cuda")
    h_out = stk.forward(h_in, per_layer_out=rec)
    torch.cuda.synchronize()
    s, f = stk.status()
    assert s == 0, (s, f)
    rec_np = rec.cpu().numpy().astype(np.float64)
    out_np = h_out.cpu().numpy().astype(np.float64)
    # the record's last plane is the call's output, bit for bit
    np.testing.assert_array_equal(rec_np[-1], out_np)
    return stk, rec_np


def _check_local(cfg, layers, h0, rec, stk, check_ids=True):
    worst = 0.0
    T = h0.shape[0]
    for l, w in enumerate(layers):
        h_in = h0.astype(np.float64) if l == 0 else rec[l - 1]
        r = O.block_forward(w, _block_input(h_in, w["rms_gamma"]), cfg.top_k)
        pred = h_in + r["out"]
        rms = np.sqrt(np.mean(r["out"] ** 2))
        err = np.abs(rec[l] - pred)
        bound = TOL * rms + half_ulp16(pred)
        assert (err <= bound).all(), f"layer {l}: max err {err.max():.3e}, rms {rms:.3e}"
        worst = max(worst, float(((err - half_ulp16(pred)).clip(0)).max() / rms))
        if check_ids:
            # ids exact: the gap at the GPU's own input is far above the GPU's logit error
            ids = stk.layer_routing(l, T)["ids"].cpu().numpy()
            np.testing.assert_array_equal(ids, r["ids"], err_msg=f"layer {l}")
    return worst


def test_stack_40_layers_one_call_local_and_chained():
    build.build()
    cfg = synth.PROD
    layers, h0, h_chain = _layers_and_input(cfg, 3, 40)
    stk, rec = _run_stack(cfg, layers, h0, max_tokens=1)
    worst = _check_local(cfg, layers, h0, rec, stk)
    chained = np.abs(rec[-1] - h_chain).max() / np.sqrt(np.mean(h_chain ** 2))
    print(f"40-layer stack (one call): worst local err/RMS beyond the fp16 residual rounding {worst:.3e}; "
          f"chained max err/RMS(h) {chained:.3e}")
    stk.close()


@pytest.mark.parametrize("T,n_layers", [(3, 3), (40, 2)])
def test_stack_multi_token_per_layer_record(T, n_layers):
    """The per-layer record from the multi-token decode kernel (T = 3) and from the prompt-chunk path (T = 40,
    copied after each layer)."""
    build.build()
    cfg = synth.PROD
    layers, h0, _ = _layers_and_input(cfg, 11 + T, n_layers, T=T)
    stk, rec = _run_stack(cfg, layers, h0, max_tokens=T)
    worst = _check_local(cfg, layers, h0, rec, stk)
    print(f"stack T={T}, {n_layers} layers: worst local err/RMS beyond the fp16 residual rounding {worst:.3e}")
    stk.close()
