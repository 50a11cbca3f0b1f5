"""Prompt-chunk configuration: one production-width block on T = 512 tokens, uniform routing and Zipf(1.1)
routing (per-expert token groups from a few tokens up to hundreds). Expert ids bit-exact, outputs within
2e-3 * RMS(out_oracle) beyond the fp16 output's own rounding (tests._cases.check_tol), plus the block gates of
the Chimera notebook."""
import numpy as np
import pytest

import oracle.moe_oracle as O
from tests._cases import check_tol, make_case, rel_err, structural
from w4a16_top_mixture_gb300 import build, lib, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 2e-3


@pytest.mark.parametrize("T,routing", [(40, "uniform"), (512, "uniform"), (512, "zipf")])
def test_chunk(T, routing):
    import torch
    build.build()
    cfg = synth.PROD
    w, x = make_case(cfg, T, 41 + T if routing == "uniform" else 42, routing=routing)
    r = O.block_forward(w, x, cfg.top_k)
    counts = np.bincount(r["ids"].ravel(), minlength=cfg.n_experts)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    s, f = blk.status()
    assert s == 0, (s, f)
    got = out.cpu().numpy().astype(np.float64)
    rt = blk.last_routing(T)
    np.testing.assert_array_equal(rt["ids"].cpu().numpy(), r["ids"])
    np.testing.assert_allclose(rt["w"].cpu().numpy(), r["w"], rtol=0, atol=2e-5)
    ok, e, plain = check_tol(got, r["out"])
    cos, ratio, moved = structural(got, r)
    print(f"T={T} {routing}: largest expert group {counts.max()}, experts used {np.count_nonzero(counts)}, "
          f"err beyond fp16 rounding/RMS = {e:.3e} (plain {plain:.3e}), cos {cos:.6f}")
    assert ok, (e, plain)
    assert cos >= 0.999 and abs(ratio - 1) <= 0.02 and moved >= 0.5
    assert blk.last_launch_count() == 8          # the tensor-core chunk path, not the decode loop
    if routing == "zipf":
        assert counts.max() >= 64          # a head expert reaches a dense-tile-sized group
    blk.close()
