"""A block loaded from the affine checkpoint layout (moe_block_load_affine) on the GPU: its outputs are bit for
bit those of the same block loaded from the expected canonical arrays (tests/_affine.py, the numpy reference of
the conversion), and match the oracle on those arrays, through the decode kernels and the prompt-chunk path."""
import numpy as np
import pytest

import oracle.moe_oracle as O
from tests._affine import make_affine
from tests._cases import check_tol
from w4a16_top_mixture_gb300 import build, lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    lib.load_library()


@pytest.mark.parametrize("dtype,small_bits", [("bf16", 8), ("f16", 4)])
def test_affine_load_equals_canonical_load(dtype, small_bits):
    import torch
    cfg = synth.TINY
    aff, exp = make_affine(cfg, 21 + small_bits, dtype, small_bits)
    blk_a = lib.MoeBlock.from_config(cfg, max_tokens=40)
    blk_a.load_affine(aff)
    blk_c = lib.MoeBlock.from_config(cfg, max_tokens=40)
    blk_c.load_weights(exp)
    rng = np.random.default_rng(31)
    for T in (1, 3, 40):
        x = rng.standard_normal((T, cfg.hidden)).astype(np.float16)
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
        out_a = blk_a.forward(xd)
        out_c = blk_c.forward(xd)
        torch.cuda.synchronize()
        assert blk_a.status()[0] == 0 and blk_c.status()[0] == 0
        a = out_a.cpu().numpy()
        np.testing.assert_array_equal(a.view(np.uint16), out_c.cpu().numpy().view(np.uint16))
        r = O.block_forward(exp, x, cfg.top_k)
        ok, e, plain = check_tol(a.astype(np.float64), r["out"])
        assert ok, (T, e, plain)
    blk_a.close()
    blk_c.close()
