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


def _sampled_check(cfg, w, x, got, ids_gpu, n_sample, seed):
    """Every token's ids against the oracle's routing of the full batch; the outputs of a seeded sample of
    tokens against the oracle run on those tokens alone (tokens are independent)."""
    Wr = O.dequant_int8(w["router_q"], w["router_s"], w["router_b"])
    lg = x.astype(np.float64) @ Wr.T
    ids, _, _ = O.route(lg[:, :cfg.n_experts], cfg.top_k)
    np.testing.assert_array_equal(ids_gpu, ids)
    pick = np.sort(np.random.default_rng(seed).choice(x.shape[0], n_sample, replace=False))
    r = O.block_forward(w, x[pick], cfg.top_k)
    ok, e, plain = check_tol(got[pick], r["out"])
    return ok, e, plain


@pytest.mark.parametrize("T", [2048, 4096])
def test_chunk_full_size_sampled(T):
    """The largest chunks the library accepts (max_tokens up to 4096): all ids, a sample of outputs."""
    import torch
    build.build()
    cfg = synth.PROD
    w, x = make_case(cfg, T, 60 + T)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    s, f = blk.status()
    assert s == 0, (s, f)
    ok, e, plain = _sampled_check(cfg, w, x, out.cpu().numpy().astype(np.float64),
                                  blk.last_routing(T)["ids"].cpu().numpy(), 16, T)
    print(f"T={T}: sampled err beyond fp16 rounding/RMS = {e:.3e} (plain {plain:.3e})")
    assert ok, (e, plain)
    blk.close()


@pytest.mark.parametrize("T", [17, 40, 200])
def test_chunk_tiny_shape(T):
    import torch
    build.build()
    cfg = synth.TINY
    w, x = make_case(cfg, T, 70 + T)
    r = O.block_forward(w, x, cfg.top_k)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    assert blk.status()[0] == 0
    assert blk.last_launch_count() == 8
    np.testing.assert_array_equal(blk.last_routing(T)["ids"].cpu().numpy(), r["ids"])
    ok, e, plain = check_tol(out.cpu().numpy().astype(np.float64), r["out"])
    assert ok, (e, plain)
    blk.close()


def test_chunk_ragged_517():
    import torch
    build.build()
    cfg = synth.PROD
    T = 517
    w, x = make_case(cfg, T, 80)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    assert blk.status()[0] == 0
    ok, e, plain = _sampled_check(cfg, w, x, out.cpu().numpy().astype(np.float64),
                                  blk.last_routing(T)["ids"].cpu().numpy(), 24, T)
    assert ok, (e, plain)
    blk.close()


def test_chunk_split_is_byte_equal():
    """A chunk split in two gives every token the same output bytes (each token's products, folds and combine
    are its own: TensorFold #3239, "Seams", chunked against token-by-token equality)."""
    import torch
    build.build()
    cfg = synth.PROD
    w, x = make_case(cfg, 512, 90)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=512)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    whole = blk.forward(xd).cpu().numpy()
    a = blk.forward(xd[:256].contiguous()).cpu().numpy()
    b = blk.forward(xd[256:].contiguous()).cpu().numpy()
    torch.cuda.synchronize()
    assert blk.status()[0] == 0
    np.testing.assert_array_equal(whole.view(np.uint16), np.concatenate([a, b]).view(np.uint16))
    blk.close()


def test_chunk_alternating_sizes_are_byte_equal():
    """Chunk forwards of two sizes alternating on one handle give the same bytes every time. (While a
    dequantisation group could wait for a stage's next fill before its previous fill had landed, a barrier-parity
    false positive, about one forward in a few hundred to a hundred computed a CTA's first down-projection job
    from a stage whose copy had not landed; start-up timing, which changes with the size, set the rate.)"""
    import torch
    build.build()
    cfg = synth.PROD
    w, x = make_case(cfg, 512, 90)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=512)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    xa = xd[:256].contiguous()
    ref_w = ref_a = None
    for _ in range(60):
        o_w = blk.forward(xd).cpu().numpy().view(np.uint16)
        o_a = blk.forward(xa).cpu().numpy().view(np.uint16)
        if ref_w is None:
            ref_w, ref_a = o_w.copy(), o_a.copy()
            np.testing.assert_array_equal(ref_w[:256], ref_a)
        np.testing.assert_array_equal(o_w, ref_w)
        np.testing.assert_array_equal(o_a, ref_a)
    torch.cuda.synchronize()
    assert blk.status()[0] == 0
    blk.close()


@pytest.mark.parametrize("T", [517, 600])
def test_chunk_repeats_are_byte_equal(T):
    """The same chunk forwarded again and again on one handle gives the same bytes every time: the GEMM's
    handoffs leave no room for timing to change a result. (When two threads of a CTA issued the MMAs, about one
    forward in thirty at these sizes had one job computed wrongly; 24 repeats of two shapes would have shown it
    with high probability.)"""
    import torch
    build.build()
    cfg = synth.PROD
    w, x = make_case(cfg, T, 80)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    first = blk.forward(xd).cpu().numpy().view(np.uint16).copy()
    for rep in range(23):
        again = blk.forward(xd).cpu().numpy().view(np.uint16)
        bad = np.nonzero((again != first).any(axis=1))[0]
        assert len(bad) == 0, (rep, bad[:16].tolist())
    assert blk.status()[0] == 0
    blk.close()


def test_chunk_bounded_wait_reports_timeout_and_recovers():
    """A withheld weight copy (host-set test flag) makes one CTA's bounded waits of the chunk GEMM run out: the
    call ends, the status reports the timeout, and the next call on the same handle is correct again. No GPU
    fault."""
    import torch
    build.build()
    cfg = synth.PROD
    T = 40
    w, x = make_case(cfg, T, 95)
    r = O.block_forward(w, x, cfg.top_k)
    blk = lib.MoeBlock.from_config(cfg, max_tokens=T)
    blk.load_weights(lib.upload_weights(w))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    blk.set_wait(timeout_us=20000, skip_arrive=True)
    blk.forward(xd)
    s, flags = blk.status()
    assert s == -5 and (flags & 512), (s, flags)
    blk.set_wait(0, False)
    out = blk.forward(xd)
    torch.cuda.synchronize()
    assert blk.status()[0] == 0
    ok, e, plain = check_tol(out.cpu().numpy().astype(np.float64), r["out"])
    assert ok, (e, plain)
    blk.close()
