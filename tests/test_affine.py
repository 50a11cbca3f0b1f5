"""The library's conversion of the affine checkpoint layout into the canonical one (moe_affine_convert, host
code, no GPU), against the independent numpy packing and conversion of tests/_affine.py: codes byte for byte,
scales and biases bit for bit, the shared gate row's quantisation exactly; and the documented refusals."""
import numpy as np
import pytest

from tests._affine import make_affine, pack_words, quantise_gate_row, to_bf16, unpack_int4_bytes
from w4a16_top_mixture_gb300 import build, lib, synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    lib.load_library()


def test_packing_helpers_round_trip():
    rng = np.random.default_rng(1)
    c4 = rng.integers(0, 16, size=(3, 128))
    w4 = pack_words(c4, 4)
    assert w4.shape == (3, 16) and w4.dtype == np.uint32
    # the 4-bit words' bytes are the canonical int4 bytes (little-endian)
    np.testing.assert_array_equal(unpack_int4_bytes(w4.view(np.uint8)), c4)
    c8 = rng.integers(0, 256, size=(2, 64))
    np.testing.assert_array_equal(pack_words(c8, 8).view(np.uint8), c8)
    assert to_bf16(np.float32([1.0, -2.5, 3.0e-3])).tolist() == [0x3F80, 0xC020, 0x3B45]


@pytest.mark.parametrize("dtype,small_bits", [("bf16", 8), ("bf16", 4), ("f16", 8), ("f16", 4)])
def test_conversion_matches_reference(dtype, small_bits):
    cfg = synth.TINY
    aff, exp = make_affine(cfg, 11 + small_bits, dtype, small_bits)
    got = lib.affine_convert(cfg, aff)
    assert sorted(got) == sorted(exp)
    for n in exp:
        if n.endswith("_q"):
            np.testing.assert_array_equal(got[n], exp[n], err_msg=n)
        else:
            np.testing.assert_array_equal(got[n].view(np.uint16), exp[n].view(np.uint16), err_msg=n)


def test_gate_row_quantisation_bound():
    """Every value of the quantised gate row is within half a step (plus the fp16 rounding of s and b) of the
    unquantised one, and constant groups are exact."""
    rng = np.random.default_rng(5)
    v = rng.normal(0, 0.05, size=512).astype(np.float32)
    v[64:128] = np.float32(0.0125)
    q, s16, b16 = quantise_gate_row(v)
    s, b = s16.astype(np.float64), b16.astype(np.float64)
    back = (s.repeat(64) * q + b.repeat(64))
    step = s.repeat(64)
    assert (np.abs(back - v) <= step * 0.5 + 1e-3 * np.abs(v) + 1e-6).all()
    assert (back[64:128] == np.float16(0.0125)).all()


def _refused(cfg, aff):
    with pytest.raises(lib.MoeError) as e:
        lib.affine_convert(cfg, aff)
    assert e.value.status == -1


def test_refusals():
    cfg = synth.TINY
    aff, _ = make_affine(cfg, 3, "bf16", 8)
    bad = dict(aff)
    q, s, b, _ = aff["exp_gate"]
    bad["exp_gate"] = (q, s, b, 8)                 # the routed experts must be 4-bit
    _refused(cfg, bad)
    bad = dict(aff)
    bad["router"] = aff["router"][:3] + (6,)       # bits other than 4 / 8
    _refused(cfg, bad)
    bad = dict(aff)
    s2 = aff["sh_up"][1].copy()
    s2.flat[7] = 0x7FC0                            # a NaN scale
    bad["sh_up"] = (aff["sh_up"][0], s2, aff["sh_up"][2], 8)
    _refused(cfg, bad)
    bad = dict(aff)
    s3 = aff["sh_up"][1].copy()
    s3.flat[0] = to_bf16(np.float32([1.0e6]))[0]   # beyond fp16's range
    bad["sh_up"] = (aff["sh_up"][0], s3, aff["sh_up"][2], 8)
    _refused(cfg, bad)
    bad = dict(aff)
    bad["scale_dtype"] = "bf16"
    A, keep = lib._affine_struct(bad)
    A.scale_dtype = 7                              # unknown dtype
    import ctypes
    c = lib.Config(cfg.hidden, cfg.n_experts, cfg.top_k, cfg.expert_inter, cfg.shared_inter, 64, 1)
    W = lib.Weights()
    assert lib.load_library().moe_affine_convert(ctypes.byref(c), ctypes.byref(A), ctypes.byref(W)) == -1
