"""The range-checking build (libbsgg_debug.so, compiled with BSGG_DEBUG_BOUNDS):
every TMA box origin, output index and scale-factor offset the kernel uses is
checked on the device against the problem's extents before the access.  Small
parity cases -- every tile shape, MXFP8 and NVFP4 inputs, ragged and empty
groups, K and N tails, row and column quantized outputs, float outputs with
amax -- run through it with no check failing and match the oracle.  A test
margin makes the row checks stricter than the buffers, so that the checks
fire on accesses that are in fact in range: the status reads
BSGG_ERR_DEVICE_BOUNDS with the failing site, and the next launch without the
margin is clean."""
import numpy as np
import pytest

import block_scaled_grouped_gb300 as bsgg
from helpers import oracle_run, small_problem
from gpu_harness import TILES, tile_id, compare, run_gpu, to_device

pytestmark = pytest.mark.gpu

CASES = {
    "gate_bf16_ragged_ktail": dict(counts=(70, 0, 130, 20), k=416, n=96, pad_to=128, seed=51),
    "swiglu_e4m3_col": dict(counts=(130, 256, 40), k=384, n=512, pad_to=128, epi="swiglu", out_fmt="e4m3",
                            want_col=True, seed=52),
    "srelu_e2m1_nvfp4": dict(counts=(0, 200, 70), k=288, n=256, pad_to=128, in_fmt="nvfp4", epi="srelu",
                             out_fmt="e2m1", tanh_clamp_s=8.0, seed=53),
    "srelu_e2m1_mxfp4_col": dict(counts=(256, 70), k=512, n=256, pad_to=128, in_fmt="mxfp4", epi="srelu",
                                out_fmt="e2m1", want_col=True, seed=54),
}


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    from block_scaled_grouped_gb300 import build as bsgg_build
    bsgg_build.build(debug_bounds=True)
    assert bsgg.lib(debug_bounds=True).bsgg_debug_bounds_checked() == 1


def _plan(p, tile):
    return bsgg.Plan(debug_bounds=True, m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups,
                     in_format=p.in_fmt, out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col,
                     tanh_clamp_s=p.tanh_clamp_s, tile=tuple(tile[:2]), cluster=tuple(tile[2:4]))


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
@pytest.mark.parametrize("case", sorted(CASES))
def test_no_check_fails_and_results_match_the_oracle(case, tile):
    p = to_device(small_problem(**CASES[case]))
    ref = oracle_run(p)
    plan = _plan(p, tile)
    outs, _, _ = run_gpu(p, plan=plan)          # asserts a clean device status
    compare(p, outs, ref)
    if "amax" in outs:
        np.testing.assert_allclose(outs["amax"].cpu().numpy(), ref["amax"], rtol=2.0 ** -10, atol=0)
    assert plan.debug_bounds_violation() == (0, 0, 0)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_a_stricter_row_limit_makes_the_checks_fire(tile):
    p = to_device(small_problem(**CASES["swiglu_e4m3_col"]))
    plan = _plan(p, tile)
    plan.debug_bounds_margin(128)               # rows >= m_pad - 128 now fail their checks
    with pytest.raises(AssertionError, match="device status 7"):
        run_gpu(p, plan=plan)
    site, value, limit = plan.debug_bounds_violation()
    assert site in (1, 10), site                # A rows (operand loads) or D rows (stores)
    assert limit == p.m_pad - 128 and limit <= value < p.m_pad, (value, limit)
    plan.debug_bounds_margin(0)
    ref = oracle_run(p)
    outs, _, _ = run_gpu(p, plan=plan)
    compare(p, outs, ref)
