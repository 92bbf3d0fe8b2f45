"""Pins for the oracle's number formats (decode tables and encoders).

The decode tables are checked exhaustively against torch's own float8
conversions (a library routine, independent of the oracle), the E2M1 table
against the format's listed values, and the encoders against torch casts, the
math library and the round-to-nearest-even definition on ties.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc


def _torch_decode(dtype):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(dtype).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt,dtype", [(orc.F_E4M3, torch.float8_e4m3fn),
                                       (orc.F_E5M2, torch.float8_e5m2)])
def test_fp8_decode_matches_torch(fmt, dtype):
    ref = _torch_decode(dtype)
    got = np.array([orc.decode(fmt, c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(got[~both_nan], ref[~both_nan])


def test_fp8_landmarks():
    # Largest finite values are the q_max of "Grouped GEMM + Quant (SM100)",
    # Equations, Step 3: 448 for E4M3 and 57344 for E5M2.
    assert orc.decode(orc.F_E4M3, 0x7E) == 448.0
    assert math.isnan(orc.decode(orc.F_E4M3, 0x7F))
    assert orc.decode(orc.F_E5M2, 0x7B) == 57344.0
    assert math.isinf(orc.decode(orc.F_E5M2, 0x7C))
    assert orc.decode(orc.F_E4M3, 0x38) == 1.0
    assert orc.decode(orc.F_E4M3, 0x01) == 2.0 ** -9


def test_ue8m0_decode_matches_torch():
    ref = _torch_decode(torch.float8_e8m0fnu)
    got = np.array([orc.decode(orc.F_UE8M0, c) for c in range(256)])
    assert math.isnan(got[255]) and math.isnan(ref[255])
    # torch materialises 2^-127 as a float64 exactly
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0


def test_e2m1_decode_is_the_listed_values():
    listed = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = [orc.decode(orc.F_E2M1, c) for c in range(16)]
    assert got[:8] == listed
    assert got[8:] == [-x for x in listed]
    assert math.copysign(1.0, got[8]) == -1.0


@pytest.mark.parametrize("fmt,dtype,qmax", [(orc.F_E4M3, torch.float8_e4m3fn, 448.0),
                                            (orc.F_E5M2, torch.float8_e5m2, 57344.0)])
def test_fp8_encode_rne_matches_torch_cast(fmt, dtype, qmax):
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(3000) * s for s in (1e-3, 0.1, 1.0, 30.0, qmax / 4)]
    x = np.concatenate(vals).astype(np.float32)
    # exact midpoints between neighbouring finite codes: ties must go to even
    pos = np.array([orc.decode(fmt, c) for c in range(0, 0x7F if fmt == orc.F_E4M3 else 0x7C)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, [0.0, -0.0]]).astype(np.float32)
    x = np.clip(x, -qmax, qmax)
    ref = torch.from_numpy(x).to(dtype).view(torch.uint8).numpy()
    got = np.array([orc.encode_rne_satfinite(fmt, float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_fp8_encode_saturates():
    assert orc.encode_rne_satfinite(orc.F_E4M3, 1e9) == 0x7E
    assert orc.encode_rne_satfinite(orc.F_E4M3, -470.0) == 0xFE
    assert orc.encode_rne_satfinite(orc.F_E4M3, float("inf")) == 0x7E
    assert orc.encode_rne_satfinite(orc.F_E5M2, 1e9) == 0x7B


def test_e2m1_encode_ties_and_saturation():
    # Round to nearest, ties to the even code (last mantissa bit 0).
    cases = {0.0: 0, 0.2: 0, 0.25: 0, 0.26: 1, 0.75: 2, 1.25: 2, 1.3: 3, 1.75: 4,
             2.5: 4, 2.6: 5, 3.5: 6, 4.9: 6, 5.0: 6, 5.1: 7, 6.0: 7, 100.0: 7}
    for x, c in cases.items():
        assert orc.encode_rne_satfinite(orc.F_E2M1, x) == c, x
        assert orc.encode_rne_satfinite(orc.F_E2M1, -x) == (c | 8), -x


def test_e2m1_encode_is_nearest_value():
    rng = np.random.default_rng(1)
    vals = np.array([orc.decode(orc.F_E2M1, c) for c in range(8)])
    for x in rng.uniform(-7, 7, 2000).astype(np.float32):
        c = orc.encode_rne_satfinite(orc.F_E2M1, float(x))
        got = orc.decode(orc.F_E2M1, c)
        best = np.min(np.abs(vals - min(abs(x), 6.0)))
        assert abs(abs(got) - min(abs(float(x)), 6.0)) == pytest.approx(best, abs=0)


def test_ue8m0_ceil_encoder():
    # exact powers of two encode to themselves
    for e in range(-126, 128):
        assert orc.encode_ue8m0_ceil(2.0 ** e) == e + 127
    # anything above a power of two rounds up (math.log2 as the independent check)
    rng = np.random.default_rng(2)
    for x in np.exp(rng.uniform(-60, 60, 2000)).astype(np.float32):
        x = float(x)
        want = math.ceil(math.log2(x))
        if 2.0 ** want < x:          # guard log2 rounding at exact powers
            want += 1
        if 2.0 ** (want - 1) >= x:
            want -= 1
        assert orc.encode_ue8m0_ceil(x) == want + 127
    assert orc.encode_ue8m0_ceil(0.0) == 0
    assert orc.encode_ue8m0_ceil(3.0e38) == 254
    assert orc.decode(orc.F_UE8M0, orc.encode_ue8m0_ceil(8.0 / 448.0)) == 2.0 ** -5
