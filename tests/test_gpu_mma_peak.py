"""The peak-measurement utility: it runs, returns a plausible dense rate
(between a quarter of and twice the nominal 4.5 / 9 PFLOP/s of MXFP8 / NVFP4
on GB300), and NVFP4 (K=64 per instruction) runs faster than MXFP8 (K=32), in
both instruction forms (cta_group::1 on single SMs, cta_group::2 on SM pairs)."""
import pytest

import block_scaled_grouped_gb300 as bsgg

pytestmark = pytest.mark.gpu


def test_mma_peak_is_plausible():
    f8 = bsgg.measure_mma_peak("mxfp8_e4m3", 256, 1 << 18)
    f4 = bsgg.measure_mma_peak("nvfp4", 256, 1 << 18)
    assert 1100.0 < f8 < 9000.0, f8
    assert 2200.0 < f4 < 18000.0, f4
    assert f4 > 1.3 * f8


def test_pair_mma_peak_is_plausible():
    f8 = bsgg.measure_mma_peak_tile("mxfp8_e4m3", 256, 256, 1 << 18)
    f4 = bsgg.measure_mma_peak_tile("nvfp4", 256, 256, 1 << 18)
    assert 1100.0 < f8 < 9000.0, f8
    assert 2200.0 < f4 < 18000.0, f4
    assert f4 > 1.3 * f8


def test_mma_peak_rejects_bad_arguments():
    with pytest.raises(bsgg.BsggError):
        bsgg.measure_mma_peak("mxfp8_e4m3", 192, 1 << 10)
    with pytest.raises(bsgg.BsggError):
        bsgg.measure_mma_peak("mxfp8_e4m3", 256, 1 << 23)
