"""Pins for the oracle's rowwise Hadamard output ("Grouped GEMM + GLU +
Hadamard + Quant (SM100)", Equations: a fixed 16-wide orthonormal Hadamard
transform of bf16-rounded D; NVFP4 RHT with E4M3 scales under rht_norm_const):

* bf16 rounding against torch's float32 -> bfloat16 cast (round to nearest even),
  ties, subnormals and large values included;
* the 16 x 16 matrix against scipy.linalg.hadamard(16) (Sylvester order);
* the transform of every 16-column block against bf16(D) @ hadamard(16) / 4
  computed with torch and scipy;
* properties: orthonormal (norm preserved), an involution, the all-ones block
  maps to (4, 0, ..., 0);
* the NVFP4 RHT: each block's E4M3 scale is RN(norm * max|y| / 6) and the codes
  dequantize within one E2M1 step of y.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle as orc
from helpers import E2M1_VALUES, np_, oracle_run, small_problem


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 2000),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130, 3 * 2.0 ** -134,
                  2.0 ** -126, 3.0e38, -3.0e38, 0.0, -0.0], dtype=np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    got = np.array([orc.round_bf16(float(v)) for v in vals])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_hadamard_matrix_is_sylvester():
    H = np.array([[orc.hadamard16(i, j) for j in range(16)] for i in range(16)])
    assert np.array_equal(H, scipy.linalg.hadamard(16))
    assert np.array_equal(H @ H.T, 16 * np.eye(16))


@pytest.mark.parametrize("epi,out_fmt", [("gate", "f32"), ("swiglu", "bf16"), ("srelu", "e4m3")])
def test_rht_blocks_against_brute_force(epi, out_fmt):
    p = small_problem(counts=(40, 0, 70), k=128, n=128, epi=epi, out_fmt=out_fmt, pad_to=32, seed=8)
    out = oracle_run(p, rht="bf16")
    d = out["d_ref"]
    xb = np.vectorize(orc.round_bf16)(d)         # bf16 rounding of the fp64 D
    H = scipy.linalg.hadamard(16) / 4.0
    want = (xb.reshape(d.shape[0], -1, 16) @ H.T).reshape(d.shape)
    np.testing.assert_allclose(out["rht_ref"], want, rtol=1e-14, atol=1e-300)
    # orthonormal: every block keeps its norm; applying H again gives bf16(D) back
    blk = out["rht_ref"].reshape(d.shape[0], -1, 16)
    np.testing.assert_allclose(np.sum(blk ** 2, -1), np.sum(xb.reshape(blk.shape) ** 2, -1), rtol=1e-12)
    scale = np.abs(xb.reshape(blk.shape)).max(-1, keepdims=True)
    back = (blk @ H.T)
    assert np.all(np.abs(back - xb.reshape(blk.shape)) <= 1e-12 * scale)


def test_all_ones_block():
    # gate with C = bias = 1 on every column (A = 0), prob 1: D = 1 -> y = (4, 0, ...)
    p = small_problem(counts=(32,), k=32, n=32, epi="gate", out_fmt="f32", pad_to=32, seed=9)
    p.a = torch.zeros_like(p.a)
    p.prob = torch.ones(32)
    out = oracle_run(p, rht="bf16", bias=np.ones((1, 32), dtype=np.float32))
    y = out["rht_ref"].reshape(32, 2, 16)
    assert np.all(y[..., 0] == 4.0) and np.all(y[..., 1:] == 0.0)


@pytest.mark.parametrize("norm", [1.0, 0.25])
def test_nvfp4_rht_quantization(norm):
    p = small_problem(counts=(64, 20), k=128, n=256, epi="swiglu", out_fmt="bf16", pad_to=32, seed=10)
    out = oracle_run(p, rht="e2m1", rht_norm=norm)
    y = out["rht_ref"]
    nd = y.shape[1]
    kb = nd // 16
    codes = out["rht_q"].reshape(p.m_pad, nd // 2)
    nib = np.stack([codes & 0xF, codes >> 4], -1).reshape(p.m_pad, nd)
    for r in range(0, p.m_pad, 5):
        for b in range(kb):
            code = int(out["sfrht"][orc.sf_offset(r, b, 0, p.m_pad, kb)])
            blk = y[r, 16 * b:16 * b + 16]
            am = float(np.abs(blk).astype(np.float32).max())
            sf = np.float32(np.float32(norm) * np.float32(am)) * np.float32(1.0 / 6.0)
            want = int(torch.tensor([float(sf)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
            assert code == want
            if am == 0:
                continue
            sfd = float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).double()[0])
            deq = E2M1_VALUES[nib[r, 16 * b:16 * b + 16]] * sfd / norm
            # within half the largest E2M1 gap (2, between 4 and 6) at the block's
            # scale, plus the saturation an E4M3 scale rounded down can cause
            assert np.all(np.abs(deq - blk) <= sfd / norm + 0.07 * am)


def test_colwise_rht_per_expert_transposed():
    """Colwise RHT: for every column and every 16-token block of an expert, the
    transform along the tokens (scipy's hadamard(16) / 4 of bf16(D)), quantized
    to NVFP4 with one E4M3 scale per block, stored per expert as the (n_d,
    expert_m) matrix with tokens contiguous at flat element n_d * start_g, and
    the scales as swizzled SF(n_d, expert_m) at byte n_d * start_g / 16."""
    p = small_problem(counts=(64, 0, 100, 64), k=128, n=256, epi="srelu", out_fmt="bf16", pad_to=64, seed=11)
    norm = 0.5
    out = oracle_run(p, rht="col_e2m1", rht_norm=norm)
    d = out["d_ref"]
    nd = d.shape[1]
    off = np_(p.padded_offsets)
    H = scipy.linalg.hadamard(16) / 4.0
    xb = np.vectorize(orc.round_bf16)(d)
    nib = np.stack([out["rht_q"] & 0xF, out["rht_q"] >> 4], -1).reshape(-1)
    start = 0
    for g in range(p.num_groups):
        em = int(off[g]) - start
        for t0 in range(0, em, 16):
            blk = xb[start + t0:start + t0 + 16]              # (16 tokens, nd)
            y = H @ blk                                        # per column, along the tokens
            np.testing.assert_allclose(out["rht_ref"][start + t0:start + t0 + 16], y, rtol=1e-14, atol=1e-300)
            for n in (0, 1, nd // 2, nd - 1):
                code = int(out["sfrht"][nd * start // 16 + orc.sf_offset(n, t0 // 16, 0, nd, em // 16)])
                am = float(np.abs(y[:, n]).astype(np.float32).max())
                sf = np.float32(np.float32(norm) * np.float32(am)) * np.float32(1.0 / 6.0)
                assert code == int(torch.tensor([float(sf)]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
                if am == 0:
                    continue
                sfd = float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).double()[0])
                e0 = nd * start + n * em + t0                  # flat element of (n, t0)
                deq = E2M1_VALUES[nib[e0:e0 + 16]] * sfd / norm
                assert np.all(np.abs(deq - y[:, n]) <= sfd / norm + 0.07 * am)
        start = int(off[g])


def test_colwise_rht_needs_64_row_groups_and_128_columns():
    p = small_problem(counts=(32, 64), k=64, n=256, epi="srelu", out_fmt="bf16", pad_to=32, seed=12)
    with pytest.raises(ValueError):
        oracle_run(p, rht="col_e2m1")
