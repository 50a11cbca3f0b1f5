"""Host-side checks of the fused decode kernel's launch planning (no GPU): every token count the decode path
serves gets a plan that fits the device's shared memory, for both block shapes the library has kernels for,
and shapes or sizes without a plan are refused with the documented status."""
import ctypes

import pytest

from w4a16_top_mixture_gb300 import build, lib, synth

SMS, SMEM = 152, 232448          # GB300: SMs, opt-in shared memory per block (bytes)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    lib.load_library()


@pytest.mark.parametrize("cfg", [synth.PROD, synth.TINY], ids=["prod", "tiny"])
def test_every_decode_token_count_has_a_plan(cfg):
    stage_bytes = set()
    for T in range(1, 17):
        st, pl = lib.decode_plan(cfg, T, SMS, SMEM)
        assert st == 0, (T, st)
        assert pl["grid"] == SMS
        assert pl["stage_bytes"] % 128 == 0
        assert 4 <= pl["stages"] <= 24
        assert pl["stages"] * pl["stage_bytes"] <= pl["smem"] <= SMEM
        # the multi-token kernel reads each pair's h from L2 (the single-token kernel stages them itself)
        assert pl["h_staged"] == 0
        stage_bytes.add(pl["stage_bytes"])
    # one stage size (8 gate/up units) for every token count
    assert len(stage_bytes) == 1
    unit = 2 * (cfg.hidden // 2 + cfg.hidden // 64 * 4)   # one int4 gate row + up row with their (s, b) pairs
    assert stage_bytes.pop() >= 8 * unit


def test_token_counts_beyond_the_decode_path_are_refused():
    assert lib.decode_plan(synth.PROD, 17, SMS, SMEM)[0] == -2
    assert lib.decode_plan(synth.PROD, 0, SMS, SMEM)[0] == -1


def test_too_few_sms_or_too_little_shared_memory_is_refused():
    # 32 SMs would give each CTA 64 output rows, above the kernel's per-CTA row limit
    assert lib.decode_plan(synth.PROD, 1, 32, SMEM)[0] == -2
    assert lib.decode_plan(synth.PROD, 1, SMS, 64 * 1024)[0] == -2
    assert lib.decode_plan(synth.PROD, 1, 0, SMEM)[0] == -1


def test_invalid_shapes_and_pointers():
    L = lib.load_library()
    bad = lib.Config(2048, 256, 8, 512, 512, 32, 16)         # group size other than 64
    out = (ctypes.c_int32 * 5)()
    assert L.moe_debug_decode_plan(ctypes.byref(bad), 1, SMS, SMEM, out) == -2
    ok = lib.Config(2048, 256, 8, 512, 512, 64, 16)
    assert L.moe_debug_decode_plan(ctypes.byref(ok), 1, SMS, SMEM, None) == -1
    assert L.moe_debug_decode_plan(None, 1, SMS, SMEM, out) == -1
