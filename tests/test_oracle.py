"""Pins of the float64 oracle against things other than itself: hand-derived fixtures, closed forms, library
routines on special cases, invariants and a scalar brute force on tiny inputs. A planted-mistake suite at the
end checks that each plausible slip in the oracle (nibble order, scale/bias swap, missing renormalisation,
wrong group index, transposed operand, gate/up swap) makes at least one pin fail."""
import contextlib
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle.moe_oracle as O
from oracle import brute
from tests._golden import codes, floats, read_kv
from w4a16_top_mixture_gb300 import synth

# ---------------------------------------------------------------- pins (each takes the oracle module `o`)


def pin_dequant_int4_golden(o):
    g = read_kv("dequant_int4_g64.txt")
    packed = np.array([int(t, 16) for t in g["bytes"].split()], np.uint8)[None, :]
    s = floats(g["scales"]).astype(np.float16)[None, :]
    b = floats(g["biases"]).astype(np.float16)[None, :]
    got = o.dequant_int4(packed, s, b)[0]
    np.testing.assert_array_equal(got, floats(g["expect"]))


def pin_dequant_int8_golden(o):
    g = read_kv("dequant_int8_g64.txt")
    q = np.stack([codes(g["row0_codes"], 64), codes(g["row1_codes"], 64)]).astype(np.uint8)
    s = np.array([[float(g["row0_scale"])], [float(g["row1_scale"])]], np.float16)
    b = np.array([[float(g["row0_bias"])], [float(g["row1_bias"])]], np.float16)
    got = o.dequant_int8(q, s, b)
    np.testing.assert_array_equal(got[0], np.arange(64) / 128.0 - 0.25)
    np.testing.assert_array_equal(got[1], np.full(64, float(g["row1_expect"])))


def pin_dequant_closed_form(o):
    """Generated int4 weights use b = -8 s, so code 8 dequantises to exactly 0 and code c to (c-8) s."""
    rng = np.random.default_rng(5)
    q, s, b = synth.int4_tensor(rng, (3,), 256)
    W = o.dequant_int4(q, s, b)
    lo = (q & 0xF).astype(np.float64)
    hi = (q >> 4).astype(np.float64)
    sf = np.repeat(s.astype(np.float64), 32, axis=-1)         # one scale per 32 bytes = 64 codes
    np.testing.assert_array_equal(W[:, 0::2], (lo - 8.0) * sf)
    np.testing.assert_array_equal(W[:, 1::2], (hi - 8.0) * sf)


def pin_routing_golden(o):
    g = read_kv("routing_e6_k3.txt")
    logits = floats(g["logits"])[None, :]
    ids, w, _ = o.route(logits, int(g["k"]))
    np.testing.assert_array_equal(ids[0], [int(t) for t in g["ids"].split()])
    np.testing.assert_allclose(w[0], floats(g["weights"]), rtol=0, atol=1e-15)
    ids1, w1, _ = o.route(logits, 1)
    assert ids1[0, 0] == int(g["k1_ids"]) and w1[0, 0] == 1.0


def pin_routing_invariants(o):
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((64, 256)) * 3
    ids, w, p = o.route(logits, 8)
    assert ids.shape == (64, 8)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (w > 0).all()
    for t in range(64):
        assert len(set(ids[t])) == 8 and list(ids[t]) == sorted(ids[t])
        sel = logits[t, ids[t]]
        rest = np.delete(logits[t], ids[t])
        assert sel.min() > rest.max()
        # closed form: renormalised top-k of the softmax = softmax of the selected logits (library routine)
        np.testing.assert_allclose(w[t], scipy.special.softmax(sel), rtol=1e-13, atol=0)
    np.testing.assert_allclose(p, scipy.special.softmax(logits, axis=-1), rtol=1e-13, atol=0)
    # brute force: full sort of every logit in Python
    for t in range(8):
        order = sorted(range(256), key=lambda e: (-logits[t, e], e))[:8]
        assert sorted(order) == list(ids[t])


def pin_activations(o):
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(o.sigmoid(z), scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(o.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(), rtol=1e-14,
                               atol=1e-300)
    assert o.sigmoid(np.array(0.0)) == 0.5 and o.silu(np.array(0.0)) == 0.0


def pin_rmsnorm(o):
    rng = np.random.default_rng(3)
    h = rng.standard_normal((4, 512))
    gam = rng.uniform(0.9, 1.1, 512)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (512,), torch.from_numpy(gam), eps=1e-6).numpy()
    np.testing.assert_allclose(o.rmsnorm(h, gam, 1e-6), ref, rtol=1e-13, atol=0)
    c = 0.37
    np.testing.assert_allclose(o.rmsnorm(np.full((1, 8), c), np.ones(8), 1e-6),
                               np.full((1, 8), c / math.sqrt(c * c + 1e-6)), rtol=1e-15)


def _tiny_layer(seed=0):
    cfg = synth.TINY
    return cfg, synth.gen_layer(cfg, seed)


def pin_block_brute(o):
    """Scalar loops (byte-by-byte codes, full sort, Python sums) equal the vectorised oracle."""
    cfg, w = _tiny_layer(1)
    x = synth.gen_x(cfg, 1, seed=1)
    r = o.block_forward(w, x, cfg.top_k)
    out, ids, wts, sg = brute.block_token(w, x[0], cfg.top_k)
    assert list(r["ids"][0]) == ids
    np.testing.assert_allclose(r["w"][0], wts, rtol=1e-12)
    assert abs(r["sg"][0] - sg) < 1e-14
    np.testing.assert_allclose(r["out"][0], out, rtol=1e-9, atol=1e-9 * np.abs(out).max())


def _onehot_router(cfg, w, hot, k_spacing=1.0):
    """Router with every code constant per row and s = 1/H', b = 0, fed x = 1: logit_e = code_e * (H/H')."""
    E, H = cfg.n_experts, cfg.hidden
    q = np.zeros((E + 1, H), np.uint8)
    vals = np.arange(E) * k_spacing
    q[:E] = (vals[:, None]).astype(np.uint8)
    q[hot] = 200                      # logit gap >= 200 - (E-1) to every other expert
    q[E] = 0
    s = np.full((E + 1, H // 64), 1.0 / H, np.float16)   # H is a power of two: exact
    b = np.zeros((E + 1, H // 64), np.float16)
    w = dict(w)
    w["router_q"], w["router_s"], w["router_b"] = q, s, b
    return w


def pin_block_special_cases(o):
    cfg, w = _tiny_layer(2)
    E, H = cfg.n_experts, cfg.hidden
    x = np.ones((1, H), np.float16)
    hot = 7
    wh = _onehot_router(cfg, w, hot)
    r = o.block_forward(wh, x, cfg.top_k)
    assert hot in r["ids"][0]
    wt = dict(zip(r["ids"][0], r["w"][0]))
    assert wt.pop(hot) >= 1 - 1e-15 and max(wt.values()) < 1e-60
    # the shared-gate row is exactly zero here: g = 0, sigmoid = 1/2 exactly
    assert r["g"][0] == 0.0 and r["sg"][0] == 0.5
    # one-hot routing: the block is one dense int4 SwiGLU MLP plus half the shared MLP (torch float64)
    def mlp(qs, kind):
        Ws = [(O.dequant_int4 if kind == 4 else O.dequant_int8)(*qs[i]) for i in range(3)]
        t = torch.from_numpy(np.asarray(x, np.float64))
        Wg, Wu, Wd = (torch.from_numpy(a) for a in Ws)
        hh = torch.nn.functional.silu(torch.nn.functional.linear(t, Wg)) * torch.nn.functional.linear(t, Wu)
        return torch.nn.functional.linear(hh, Wd).numpy()[0]
    ye = mlp([(w[n + "_q"][hot], w[n + "_s"][hot], w[n + "_b"][hot]) for n in ("exp_gate", "exp_up", "exp_down")], 4)
    ys = mlp([(w[n + "_q"], w[n + "_s"], w[n + "_b"]) for n in ("sh_gate", "sh_up", "sh_down")], 8)
    np.testing.assert_allclose(r["out"][0], ye + 0.5 * ys, rtol=1e-12, atol=1e-12 * np.abs(ye).max())


def pin_block_all_experts(o):
    """k = E: top-k and renormalisation drop out and the block is the dense softmax mixture of every expert."""
    cfg, w = _tiny_layer(3)
    x = synth.gen_x(cfg, 3, seed=3).astype(np.float64)
    r = o.block_forward(w, x, cfg.n_experts)
    E = cfg.n_experts
    Wr = O.dequant_int8(w["router_q"], w["router_s"], w["router_b"])
    lg = x @ Wr.T
    pr = scipy.special.softmax(lg[:, :E], axis=-1)
    ys = []
    for e in range(E):
        Wg = O.dequant_int4(w["exp_gate_q"][e], w["exp_gate_s"][e], w["exp_gate_b"][e])
        Wu = O.dequant_int4(w["exp_up_q"][e], w["exp_up_s"][e], w["exp_up_b"][e])
        Wd = O.dequant_int4(w["exp_down_q"][e], w["exp_down_s"][e], w["exp_down_b"][e])
        ys.append(((x @ Wg.T) * scipy.special.expit(x @ Wg.T) * (x @ Wu.T)) @ Wd.T)
    Y = np.stack(ys, 1)                                      # [T, E, H]
    routed = np.einsum("te,teh->th", pr, Y)
    np.testing.assert_allclose(r["routed"], routed, rtol=1e-10, atol=1e-10 * np.abs(routed).max())


def pin_expert_permutation(o):
    """Relabelling the experts (router rows and expert tensors together) leaves the output unchanged."""
    cfg, w = _tiny_layer(4)
    x = synth.gen_x(cfg, 2, seed=4)
    r0 = o.block_forward(w, x, cfg.top_k)
    E = cfg.n_experts
    perm = np.random.default_rng(9).permutation(E)
    wp = dict(w)
    for n in ("router_q", "router_s", "router_b"):
        wp[n] = np.concatenate([w[n][:E][perm], w[n][E:]], 0)
    for n in ("exp_gate", "exp_up", "exp_down"):
        for sfx in ("_q", "_s", "_b"):
            wp[n + sfx] = w[n + sfx][perm]
    r1 = o.block_forward(wp, x, cfg.top_k)
    np.testing.assert_allclose(r1["out"], r0["out"], rtol=1e-12, atol=1e-12)
    inv = np.argsort(perm)
    for t in range(2):
        assert sorted(perm[r1["ids"][t]]) == list(r0["ids"][t])
        assert sorted(inv[r0["ids"][t]]) == list(r1["ids"][t])


def pin_stack_residual(o):
    """Stack of layers whose blocks are switched off (all expert and shared down codes at the zero point) is
    the identity; one live layer adds exactly its block output on the RMSNorm of its input."""
    cfg = synth.TINY
    layers = [synth.gen_layer(cfg, 7, l, with_gamma=True) for l in range(3)]
    dead = []
    for w in layers:
        d = dict(w)
        d["exp_down_q"] = np.full_like(w["exp_down_q"], 0x88)    # both nibbles 8: (8-8)*s = 0
        d["sh_down_q"] = np.full_like(w["sh_down_q"], 128)       # (128-128)*s = 0
        dead.append(d)
    h0 = synth.gen_x(cfg, 2, seed=7).astype(np.float64)
    hN, _ = o.stack_forward(dead, h0, cfg.top_k)
    np.testing.assert_array_equal(hN, h0)
    h1, recs = o.stack_forward([layers[0]], h0, cfg.top_k)
    xn = torch.nn.functional.rms_norm(torch.from_numpy(h0), (cfg.hidden,),
                                      torch.from_numpy(layers[0]["rms_gamma"].astype(np.float64)), eps=1e-6).numpy()
    np.testing.assert_allclose(recs[0]["x_norm"], xn, rtol=1e-13)
    np.testing.assert_allclose(h1, h0 + o.block_forward(layers[0], xn, cfg.top_k)["out"], rtol=1e-13, atol=1e-13)


PINS = [pin_dequant_int4_golden, pin_dequant_int8_golden, pin_dequant_closed_form, pin_routing_golden,
        pin_routing_invariants, pin_activations, pin_rmsnorm, pin_block_brute, pin_block_special_cases,
        pin_block_all_experts, pin_expert_permutation, pin_stack_residual]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(O)


# ---------------------------------------------------------------- planted mistakes (in the oracle, on CPU)


@contextlib.contextmanager
def planted(**repl):
    saved = {k: getattr(O, k) for k in repl}
    try:
        for k, v in repl.items():
            setattr(O, k, v)
        yield
    finally:
        for k, v in saved.items():
            setattr(O, k, v)


def _swapped_nibbles(packed):
    p = packed.astype(np.int64)
    out = np.empty((*packed.shape[:-1], 2 * packed.shape[-1]), np.int64)
    out[..., 0::2] = p >> 4
    out[..., 1::2] = p & 0xF
    return out


_orig_dequant = O.dequant
_orig_route = O.route
_orig_swiglu = O.swiglu_expert


def _dequant_swapped_sb(codes, s, b, group=64):
    return _orig_dequant(codes, b, s, group)


def _dequant_group32(codes, s, b, group=64):
    q = codes.astype(np.float64)
    idx = np.minimum(np.arange(q.shape[-1]) // 32, s.shape[-1] - 1)
    return s.astype(np.float64)[..., idx] * q + b.astype(np.float64)[..., idx]


def _route_no_renorm(logits, k):
    ids, w, p = _orig_route(logits, k)
    return ids, np.take_along_axis(p, ids, -1), p


def _route_smallest(logits, k):
    return _orig_route(-logits, k)


def _swiglu_gate_up_swapped(Wg, Wu, Wd, x):
    return _orig_swiglu(Wu, Wg, Wd, x)


def _swiglu_down_rows_reversed(Wg, Wu, Wd, x):
    y, h = _orig_swiglu(Wg, Wu, Wd, x)
    return y[:, ::-1], h


def _swiglu_sigmoid_not_silu(Wg, Wu, Wd, x):
    h = O.sigmoid(x @ Wg.T) * (x @ Wu.T)
    return h @ Wd.T, h


_orig_block = O.block_forward
_orig_rmsnorm = O.rmsnorm


def _block_shared_gate_ignored(w, x, top_k, *args, **kw):
    r = _orig_block(w, x, top_k, *args, **kw)
    r["out"] = r["routed"] + r["shared"]
    return r


def _block_shared_dropped(w, x, top_k, *args, **kw):
    r = _orig_block(w, x, top_k, *args, **kw)
    r["out"] = r["routed"].copy()
    return r


def _rmsnorm_no_gamma(h, gamma, eps=1e-6):
    return _orig_rmsnorm(h, np.ones_like(np.asarray(gamma, np.float64)), eps)


def _rmsnorm_eps_outside(h, gamma, eps=1e-6):
    h = np.asarray(h, np.float64)
    return h / (np.sqrt(np.mean(h * h, axis=-1, keepdims=True)) + eps) * np.asarray(gamma, np.float64)


def _stack_residual_dropped(layers, h0, top_k, eps=1e-6, group=64):
    h = np.asarray(h0, np.float64)
    recs = []
    for w in layers:
        xn = O.rmsnorm(h, w["rms_gamma"], eps)
        r = O.block_forward(w, xn, top_k, group)
        r["h_in"], r["x_norm"] = h, xn
        h = r["out"]
        recs.append(r)
    return h, recs


MUTANTS = {
    "shared_gate_ignored": dict(block_forward=_block_shared_gate_ignored),
    "shared_expert_dropped": dict(block_forward=_block_shared_dropped),
    "rmsnorm_no_gamma": dict(rmsnorm=_rmsnorm_no_gamma),
    "rmsnorm_eps_outside_sqrt": dict(rmsnorm=_rmsnorm_eps_outside),
    "residual_dropped": dict(stack_forward=_stack_residual_dropped),
    "nibble_order": dict(unpack_int4=_swapped_nibbles),
    "scale_bias_swap": dict(dequant=_dequant_swapped_sb),
    "group_index": dict(dequant=_dequant_group32),
    "no_renorm": dict(route=_route_no_renorm),
    "smallest_k": dict(route=_route_smallest),
    "gate_up_swap": dict(swiglu_expert=_swiglu_gate_up_swapped),
    "down_rows_reversed": dict(swiglu_expert=_swiglu_down_rows_reversed),
    "sigmoid_for_silu": dict(swiglu_expert=_swiglu_sigmoid_not_silu),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    failures = []
    with planted(**MUTANTS[name]):
        for pin in PINS:
            try:
                pin(O)
            except AssertionError:
                failures.append(pin.__name__)
    assert failures, f"planted mistake {name!r} passed every pin"
