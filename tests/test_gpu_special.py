"""The block's structural special cases through the CUDA path (the decode kernels and the prompt-chunk path),
against the oracle, which the pins tie to the same closed forms (tests/test_oracle.py):

* one-hot router: one expert's logit exceeds every other by tens, so its renormalised weight is 1 and the
  block is that expert's SwiGLU MLP plus the shared term; at production width the other experts' logits
  repeat, so exact ties also reach the top k and the lower index must win them (the oracle's reading);
* zero shared-gate row: the gate logit is exactly 0 and sigma(0) = 1/2 exactly;
* all weights exactly zero (int4 code 8 with b = -8 s, int8 code 128 with b = -128 s): with integer-valued
  activations every logit is exactly 0, the top k are the k lowest indices with weight 1/k each, and the output
  is exactly zero, bit for bit, so no stale on-chip data can leak into it.
Integer codes with s = 1/H and activations of 1 keep every logit an exact integer on the GPU too (the
kernels' 16-bit activation grid holds 1 exactly)."""
import numpy as np
import pytest

import oracle.moe_oracle as O
from tests._cases import check_tol
from w4a16_top_mixture_gb300 import build, lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    lib.load_library()


def onehot_router(cfg, w, hot):
    """Row e of the router: code c_e everywhere with s = 1/H, b = 0, so x = 1 gives logit_e = c_e exactly. The
    hot expert gets code 200; the others codes below 150 (repeating at production width); the shared-gate row
    is zero."""
    E, H = cfg.n_experts, cfg.hidden
    q = np.zeros((E + 1, H), np.uint8)
    q[:E] = (np.arange(E) * 150 // max(E, 150))[:, None].astype(np.uint8)
    q[hot] = 200
    s = np.full((E + 1, H // 64), 1.0 / H, np.float16)
    b = np.zeros((E + 1, H // 64), np.float16)
    w = dict(w)
    w["router_q"], w["router_s"], w["router_b"] = q, s, b
    return w


def zero_layer(cfg, seed):
    """Every weight exactly zero: int4 code 8 with b = -8 s, int8 code 128 with b = -128 s."""
    w = synth.gen_layer(cfg, seed)
    for n in ("exp_gate", "exp_up", "exp_down"):
        w[n + "_q"] = np.full_like(w[n + "_q"], 0x88)
    for n in ("router", "sh_gate", "sh_up", "sh_down"):
        w[n + "_q"] = np.full_like(w[n + "_q"], 128)
    return w


def _run(cfg, w, x, max_tokens):
    import torch
    blk = lib.MoeBlock.from_config(cfg, max_tokens=max_tokens)
    blk.load_weights(w)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    s, f = blk.status()
    assert s == 0, (s, f)
    rt = blk.last_routing(x.shape[0])
    res = (out.cpu().numpy(), rt["ids"].cpu().numpy(), rt["w"].cpu().numpy(), rt["sg"].cpu().numpy())
    blk.close()
    return res


CASES = [("tiny", 1), ("tiny", 3), ("tiny", 40), ("prod", 1), ("prod", 3), ("prod", 40)]


@pytest.mark.parametrize("cfgname,T", CASES)
def test_onehot_router_and_zero_gate(cfgname, T):
    cfg = synth.TINY if cfgname == "tiny" else synth.PROD
    hot = 7
    w = onehot_router(cfg, synth.gen_layer(cfg, 21), hot)
    x = np.ones((T, cfg.hidden), np.float16)
    r = O.block_forward(w, x, cfg.top_k)
    out, ids, wts, sg = _run(cfg, w, x, max_tokens=max(T, 16))
    np.testing.assert_array_equal(ids, r["ids"])           # ties at production width: lower index wins
    assert (ids == hot).any(axis=1).all()
    np.testing.assert_allclose(wts, r["w"], rtol=0, atol=1e-6)
    assert (wts[ids == hot] == 1.0).all()
    assert (sg == 0.5).all()                                # sigma of an exactly zero gate logit
    ok, e, plain = check_tol(out.astype(np.float64), r["out"])
    assert ok, (e, plain)


@pytest.mark.parametrize("cfgname,T", CASES)
def test_all_zero_weights_give_exact_zero(cfgname, T):
    cfg = synth.TINY if cfgname == "tiny" else synth.PROD
    w = zero_layer(cfg, 22)
    # integer activations keep both halves of every group's fold (s * sum(q x) and b * sum(x)) exact, so the
    # zero weights cancel exactly in fp32 as they do in float64
    x = np.random.default_rng(23).integers(-2, 3, size=(T, cfg.hidden)).astype(np.float16)
    out, ids, wts, sg = _run(cfg, w, x, max_tokens=max(T, 16))
    r = O.block_forward(w, x, cfg.top_k)
    assert (r["out"] == 0).all() and (r["ids"] == np.arange(cfg.top_k)).all()
    np.testing.assert_array_equal(ids, r["ids"])
    assert (wts == np.float32(1.0 / cfg.top_k)).all()
    assert (sg == 0.5).all()
    assert (out.view(np.uint16) == 0).all(), "output not exactly +0"


def _valid_routing(ids, E, K):
    assert ids.shape[1] == K
    assert ((ids >= 0) & (ids < E)).all(), ids
    assert (np.diff(ids, axis=1) > 0).all(), ids            # distinct and ascending


@pytest.mark.parametrize("cfgname,T", CASES)
def test_nonfinite_activations_keep_routing_in_bounds(cfgname, T):
    """A token whose activations hold NaN or an infinity makes every router logit NaN (or infinite). The top k
    must still name k distinct experts below E (everything downstream indexes by them), and the other tokens
    of the call must come out as if that token were absent."""
    import ctypes
    import torch
    cfg = synth.TINY if cfgname == "tiny" else synth.PROD
    w = synth.gen_layer(cfg, 24)
    x = synth.gen_x(cfg, T, 25)
    bad = {0: np.float16(np.nan), 1: np.float16(np.inf), 2: np.float16(-np.inf)}
    for t, v in bad.items():
        if t < T and (T == 1 or t != T - 1):                 # the last token of a multi-token call stays finite
            x[t, 5 * t + 3] = v
    nonfinite = ~np.isfinite(x.astype(np.float32)).all(axis=1)
    assert nonfinite.any() and (T == 1 or not nonfinite.all())
    out, ids, wts, sg = _run(cfg, w, x, max_tokens=max(T, 16))
    _valid_routing(ids, cfg.n_experts, cfg.top_k)
    good = np.flatnonzero(~nonfinite)
    if good.size:
        r = O.block_forward(w, x[good], cfg.top_k)
        np.testing.assert_array_equal(ids[good], r["ids"])
        ok, e, plain = check_tol(out[good].astype(np.float64), r["out"])
        assert ok, (e, plain)
    # the allocation-free routing entry point, on the same tokens
    L = lib.load_library()
    dev = {n: torch.from_numpy(np.ascontiguousarray(w[n]).view(np.uint8)).cuda() for n in
           ("router_q", "router_s", "router_b")}
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()
    ids2 = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w2 = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    sg2 = torch.empty((T,), dtype=torch.float32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    s = L.moe_router_topk_noalloc(*(ctypes.c_void_p(dev[n].data_ptr()) for n in ("router_q", "router_s", "router_b")),
                                  cfg.hidden, cfg.n_experts, cfg.top_k, ctypes.c_void_p(xd.data_ptr()), T,
                                  ctypes.c_void_p(ids2.data_ptr()), ctypes.c_void_p(w2.data_ptr()),
                                  ctypes.c_void_p(sg2.data_ptr()), st)
    assert s == 0, s
    torch.cuda.synchronize()
    ids2 = ids2.cpu().numpy()
    _valid_routing(ids2, cfg.n_experts, cfg.top_k)
    if good.size:
        np.testing.assert_array_equal(ids2[good], r["ids"])


@pytest.mark.parametrize("name,value", [("exp_down_s", 5000.0), ("sh_up_s", 300.0)])
def test_chunk_handle_refuses_out_of_range_scale(name, value):
    """A handle that serves prompt chunks forms s * q in fp16 on its chunk path: it refuses scales whose product
    with the largest code (15 for int4, 255 for int8) reaches 65504, and stays unloaded. A decode-only handle
    (max_tokens <= 16, fp32 arithmetic) takes the same weights."""
    cfg = synth.TINY
    w = synth.gen_layer(cfg, 5)
    w[name] = w[name].copy()
    w[name].flat[3] = np.float16(value)
    chunky = lib.MoeBlock.from_config(cfg, max_tokens=40)
    with pytest.raises(lib.MoeError) as e:
        chunky.load_weights(w)
    assert e.value.status == -1
    chunky.close()
    dec = lib.MoeBlock.from_config(cfg, max_tokens=16)
    dec.load_weights(w)
    dec.close()
