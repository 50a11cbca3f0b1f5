"""The seeded workloads the parity tests draw (no GPU): every token's k-th/(k+1)-th expert-logit gap under
the oracle's float64 router is at least the 1e-2 that bit-exact expert ids rely on, the draws are
reproducible, and Zipf routing concentrates tokens on few experts while uniform routing spreads them."""
import numpy as np

import oracle.moe_oracle as O
from tests._cases import MIN_GAP, gaps, make_case
from w4a16_top_mixture_gb300 import synth


def _ids_and_gaps(cfg, w, x):
    Wr = O.dequant_int8(w["router_q"], w["router_s"], w["router_b"])
    lg = x.astype(np.float64) @ Wr.T
    ids, _, _ = O.route(lg[:, :cfg.n_experts], cfg.top_k)
    return ids, gaps(lg[:, :cfg.n_experts], cfg.top_k)


def test_router_gap_respected_and_reproducible():
    cfg = synth.TINY
    for routing in ("uniform", "zipf"):
        w, x = make_case(cfg, 48, 7, routing=routing)
        ids, g = _ids_and_gaps(cfg, w, x)
        assert g.min() >= MIN_GAP, routing
        assert ids.shape == (48, cfg.top_k)
        w2, x2 = make_case(cfg, 48, 7, routing=routing)
        np.testing.assert_array_equal(x, x2)
        np.testing.assert_array_equal(w["router_q"], w2["router_q"])


def test_zipf_routing_concentrates_tokens():
    cfg = synth.TINY
    counts = {}
    for routing in ("uniform", "zipf"):
        w, x = make_case(cfg, 96, 11, routing=routing)
        ids, _ = _ids_and_gaps(cfg, w, x)
        counts[routing] = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    # the busiest expert under Zipf routing takes clearly more of the (token, slot) pairs than under uniform
    assert counts["zipf"].max() > 1.5 * counts["uniform"].max()
