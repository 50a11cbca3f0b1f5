"""The allocation-free routing entry point (moe_router_topk_noalloc) against the regular forward's routing.

It serves callers that cannot allocate device memory when they call (a serving runtime whose pool allocator
must account for every device byte, a latency-critical loop that cannot afford cudaMalloc's device-wide
synchronisation): its scratch is a fixed array inside the library. This file is collected last so that a failure
here cannot hide any other test."""
import ctypes

import numpy as np
import pytest

import oracle.moe_oracle as O
from tests._cases import make_case, quantize_acts
from w4a16_top_mixture_gb300 import build, lib, synth

pytestmark = pytest.mark.gpu


def _routing_noalloc(L, wdev, cfg, xd, T):
    import torch
    ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    sg = torch.empty((T,), dtype=torch.float32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    s = L.moe_router_topk_noalloc(ctypes.c_void_p(wdev["router_q"].data_ptr()),
                                  ctypes.c_void_p(wdev["router_s"].data_ptr()),
                                  ctypes.c_void_p(wdev["router_b"].data_ptr()), cfg.hidden, cfg.n_experts,
                                  cfg.top_k, ctypes.c_void_p(xd.data_ptr()), T, ctypes.c_void_p(ids.data_ptr()),
                                  ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(sg.data_ptr()), st)
    assert s == 0, s
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), sg.cpu().numpy()


@pytest.mark.parametrize("cfgname", ["tiny", "prod"])
def test_noalloc_routing_matches_forward_twice(cfgname):
    import torch
    build.build()
    L = lib.load_library()
    cfg = synth.TINY if cfgname == "tiny" else synth.PROD
    for call, (T, seed) in enumerate([(16, 31), (5, 32)]):
        w, x = make_case(cfg, T, seed)
        wdev = lib.upload_weights(w)
        blk = lib.MoeBlock.from_config(cfg, 16)
        blk.load_weights(wdev)
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
        blk.forward(xd)
        ref = blk.last_routing(T)
        ids, wt, sg = _routing_noalloc(L, wdev, cfg, xd, T)
        np.testing.assert_array_equal(ids, ref["ids"].cpu().numpy(), err_msg=f"call {call}")
        # this entry point computes on the fp16 activations in plain fp32, the forward on its 16-bit activation
        # grid: the tolerance is the block tests' one plus the grid's own effect, measured on the oracle
        r_x, r_q = O.block_forward(w, x, cfg.top_k), O.block_forward(w, quantize_acts(x), cfg.top_k)
        dw, dsg = np.abs(r_x["w"] - r_q["w"]).max(), np.abs(r_x["sg"] - r_q["sg"]).max()
        np.testing.assert_allclose(wt, ref["w"].cpu().numpy(), rtol=0, atol=2e-5 + dw)
        np.testing.assert_allclose(sg, ref["sg"].cpu().numpy(), rtol=0, atol=2e-6 + dsg)
        np.testing.assert_allclose(wt, r_x["w"], rtol=0, atol=2e-5)
        np.testing.assert_allclose(sg, r_x["sg"], rtol=0, atol=2e-6)
        # and both agree with the oracle's ids
        np.testing.assert_array_equal(ids, O.block_forward(w, x, cfg.top_k)["ids"])
        blk.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    build.build()
    L = lib.load_library()
    cfg = synth.TINY
    dummy = torch.zeros(1024 * 1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.moe_router_topk_noalloc(p, p, p, cfg.hidden, cfg.n_experts, cfg.top_k, p, 65, p, p, p, st) == -1
    assert L.moe_router_topk_noalloc(p, p, p, cfg.hidden, 513, 4, p, 1, p, p, p, st) == -1
    assert L.moe_router_topk_noalloc(None, p, p, cfg.hidden, cfg.n_experts, cfg.top_k, p, 1, p, p, p, st) == -1
