"""Pins for the oracle's dSwiGLU backward ("Grouped GEMM + dGLU (SM100)",
Block-scaled contract, Steps 1-3):

* the GEMM of the backward is ref = alpha_g^2 * sum_k A B (brute-force dense
  dequantization and matmul, times alpha again);
* the two gradient blocks are ref * d(forward D)/dX and ref * d(forward D)/dG,
  checked against central finite differences of the oracle's own FORWARD SwiGLU
  (pinned separately by closed forms), evaluated at chosen (X, G) by setting
  A = 0 so that C equals a chosen bias;
* dprob is the sum over GEMM columns of ref * (forward D at prob = 1);
* invariants: prob = 0 zeroes D but not dprob; beta and the saved C trade a
  power of two exactly; D and dprob are linear in ref (alpha -> 2 alpha: x4);
  block order follows gate_first; amax has an input and a gate entry per group.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import brute_force_C, np_, oracle_inputs, oracle_run, small_problem


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()


def _forward_d(xg_pairs, prob=1.0, h=0.0, which=None):
    """Forward SwiGLU D of the oracle at the given (X, G) points, C = bias (A = 0).
    `which` = "x" or "g" shifts that operand by h."""
    P = len(xg_pairs)
    n = 64 * P
    p = small_problem(counts=(32,), k=32, n=n, epi="swiglu", out_fmt="f32", pad_to=32, seed=1)
    p.a = torch.zeros_like(p.a)
    p.alpha = torch.ones(1)
    p.prob = torch.full((32,), prob, dtype=torch.float32)
    bias = np.zeros((1, n), dtype=np.float64)
    for b, (x, g) in enumerate(xg_pairs):
        bias[0, 64 * b:64 * b + 32] = x + (h if which == "x" else 0.0)
        bias[0, 64 * b + 32:64 * b + 64] = g + (h if which == "g" else 0.0)
    # the forward oracle takes a float32 bias: evaluate at float32-exact points
    ref = oracle_run(p, bias=bias.astype(np.float32))
    return ref["d_ref"][0].reshape(P, 32)[:, 0]


POINTS = [(1.0, 0.0), (0.5, 1.5), (-2.0, 0.75), (3.0, -1.25), (-0.25, -3.0), (1.5, 4.0)]


def _backward_at(points, ref_codes, alpha=1.0, prob=0.75, beta=1.0, gate_first=0):
    """Backward of the oracle with ref_n = alpha^2 * 1.0 * b_n exactly (K = 32, one
    non-zero term, unit scales) and saved C at the chosen points."""
    P = len(points)
    n = 32 * P
    p = small_problem(counts=(32,), k=32, n=n, epi="dswiglu", out_fmt="f32", pad_to=32, seed=2)
    a = torch.zeros(32, 32, dtype=torch.uint8)
    a[:, 0] = 0x38                                   # 1.0
    b = torch.zeros(1, n, 32, dtype=torch.uint8)
    b[0, :, 0] = torch.tensor(ref_codes, dtype=torch.uint8).repeat_interleave(32)   # one ref per block
    p.a, p.b = a, b
    p.sfa_rows = torch.full_like(p.sfa_rows, 127)
    p.sfb_rows = torch.full_like(p.sfb_rows, 127)
    p.alpha = torch.tensor([alpha], dtype=torch.float32)
    p.prob = torch.full((32,), prob, dtype=torch.float32)
    p.beta = torch.tensor([beta], dtype=torch.float32)
    saved = np.zeros((32, 2 * n))
    for blk, (x, g) in enumerate(points):
        xo, go = (64 * blk + 32, 64 * blk) if gate_first else (64 * blk, 64 * blk + 32)
        saved[:, xo:xo + 32] = x / beta
        saved[:, go:go + 32] = g / beta
    p.saved_c = torch.from_numpy(saved).to(torch.bfloat16)
    out = oracle_run(p, gate_first=gate_first)
    return p, out


def _e4m3_values(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


REF_CODES = [0x40, 0x38, 0xB8, 0x44, 0x30, 0xC0]    # 2, 1, -1, 3, 0.5, -2


@pytest.mark.parametrize("gate_first", [0, 1])
def test_gradients_are_finite_differences_of_the_forward(gate_first):
    pts = [(float(_bf16(x)), float(_bf16(g))) for x, g in POINTS]
    p, out = _backward_at(pts, REF_CODES, prob=0.75, gate_first=gate_first)
    ref = _e4m3_values(REF_CODES)                    # alpha = 1
    h = 2.0 ** -12
    dfdx = (_forward_d(pts, h=h, which="x") - _forward_d(pts, h=-h, which="x")) / (2 * h)
    dfdg = (_forward_d(pts, h=h, which="g") - _forward_d(pts, h=-h, which="g")) / (2 * h)
    d = out["d_ref"][0].reshape(len(pts), 64)
    din = d[:, 32] if gate_first else d[:, 0]
    dgt = d[:, 0] if gate_first else d[:, 32]
    np.testing.assert_allclose(din, ref * 0.75 * dfdx, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dgt, ref * 0.75 * dfdg, rtol=1e-6, atol=1e-9)
    # every column of a block carries the same point
    assert np.all(d[:, 0:32] == d[:, :1]) and np.all(d[:, 32:64] == d[:, 32:33])


def test_dprob_is_ref_times_forward_at_unit_prob():
    pts = [(float(_bf16(x)), float(_bf16(g))) for x, g in POINTS]
    p, out = _backward_at(pts, REF_CODES, prob=0.3)
    ref = _e4m3_values(REF_CODES)
    fwd = _forward_d(pts, prob=1.0)
    want = 32 * np.sum(ref * fwd)                    # 32 columns per block share a point
    np.testing.assert_allclose(out["dprob_ref"], np.full(32, want), rtol=1e-12)


def test_zero_prob_zeroes_d_but_not_dprob():
    pts = [(1.5, 0.5), (-1.0, 2.0)]
    p, out = _backward_at(pts, REF_CODES[:2], prob=0.0)
    assert np.all(out["d_ref"] == 0.0)
    assert np.all(np.abs(out["dprob_ref"]) > 0.0)


def test_beta_and_saved_c_trade_a_power_of_two():
    pts = [(1.5, 0.5), (-1.0, 2.0), (0.25, -0.75)]
    _, o1 = _backward_at(pts, REF_CODES[:3], beta=1.0)
    _, o2 = _backward_at(pts, REF_CODES[:3], beta=4.0)     # saved C = point / 4
    assert np.array_equal(o1["d_ref"], o2["d_ref"])
    assert np.array_equal(o1["dprob_ref"], o2["dprob_ref"])


def test_linear_in_ref_alpha_squared():
    pts = [(1.5, 0.5), (-1.0, 2.0)]
    _, o1 = _backward_at(pts, REF_CODES[:2], alpha=1.0)
    _, o2 = _backward_at(pts, REF_CODES[:2], alpha=2.0)
    assert np.array_equal(o2["d_ref"], 4.0 * o1["d_ref"])
    assert np.array_equal(o2["dprob_ref"], 4.0 * o1["dprob_ref"])


def test_closed_forms():
    # X = 1, G = 0: sigmoid 1/2, swish 0 -> d input 0, d gate = ref prob / 2, dprob 0
    # X = 2, G = ln 3: sigmoid 3/4 -> d input = ref p (3/4) ln3,
    #                  d gate = ref p 2 (3/4)(1 + ln3 / 4)
    ln3 = float(np.log(3.0))
    p, out = _backward_at([(1.0, 0.0)], [0x40], prob=0.5)           # ref = 2
    d = out["d_ref"][0]
    assert np.all(d[:32] == 0.0)
    np.testing.assert_allclose(d[32:], 2 * 0.5 * 0.5, rtol=1e-15)
    assert np.all(out["dprob_ref"] == 0.0)
    g = float(_bf16(ln3))
    p, out = _backward_at([(2.0, g)], [0x40], prob=0.5)
    s = 1.0 / (1.0 + np.exp(-g))
    np.testing.assert_allclose(out["d_ref"][0, :32], 2 * 0.5 * g * s, rtol=1e-15)
    np.testing.assert_allclose(out["d_ref"][0, 32:], 2 * 0.5 * 2 * s * (1 + g * (1 - s)), rtol=1e-15)
    assert abs(s - 0.75) < 1e-2


@pytest.mark.parametrize("in_fmt", ["mxfp8_e4m3", "nvfp4"])
def test_gemm_is_alpha_squared_brute_force(in_fmt):
    # random operands, ragged groups: every D value equals ref * (finite
    # difference of a numpy forward) with ref from the dense brute force
    p = small_problem(counts=(40, 0, 70), k=128, n=64, epi="dswiglu", out_fmt="f32", in_fmt=in_fmt,
                      pad_to=32, seed=5)
    out = oracle_run(p)
    alpha = np_(p.alpha).astype(np.float64)
    C = brute_force_C(p)                             # alpha * A B^T per group
    off = np_(p.padded_offsets)
    grp = np.searchsorted(off, np.arange(p.m_pad), side="right")
    ref = C * alpha[grp][:, None]                    # alpha^2 * A B^T
    saved = np_(p.saved_c.double()) * np_(p.beta).astype(np.float64)[grp][:, None]
    n = p.n
    bidx = np.arange(n) // 32
    ridx = np.arange(n) % 32
    X = saved[:, 64 * bidx + ridx]
    G = saved[:, 64 * bidx + 32 + ridx]

    def fwd(x, g):
        return x * g / (1.0 + np.exp(-g))
    h = 1e-6
    dx = (fwd(X + h, G) - fwd(X - h, G)) / (2 * h)
    dg = (fwd(X, G + h) - fwd(X, G - h)) / (2 * h)
    prob = np_(p.prob).astype(np.float64)[:, None]
    want = np.zeros((p.m_pad, 2 * n))
    want[:, 64 * bidx + ridx] = ref * prob * dx
    want[:, 64 * bidx + 32 + ridx] = ref * prob * dg
    scale = np.abs(want).max()
    np.testing.assert_allclose(out["d_ref"], want, rtol=1e-6, atol=1e-8 * scale)
    np.testing.assert_allclose(out["dprob_ref"], np.sum(ref * fwd(X, G), axis=1),
                               rtol=1e-9, atol=1e-9 * np.abs(ref).max())
    # amax: input-gradient and gate-gradient blocks of each group, 0 for empty
    am = out["amax"].reshape(-1, 2)
    start = 0
    for g in range(p.num_groups):
        rows = slice(start, int(off[g]))
        if off[g] > start:
            np.testing.assert_allclose(am[g, 0], np.abs(want[rows][:, 64 * bidx + ridx]).max(), rtol=1e-6)
            np.testing.assert_allclose(am[g, 1], np.abs(want[rows][:, 64 * bidx + 32 + ridx]).max(), rtol=1e-6)
        else:
            assert am[g, 0] == 0 and am[g, 1] == 0
        start = int(off[g])


def test_quantized_backward_output_is_the_step3_quantization_of_d():
    # E4M3 row and column outputs of width 2N: each block's scale is the least
    # power of two >= max|D| / 448, and codes dequantize within one step of D
    p = small_problem(counts=(64, 30), k=128, n=64, epi="dswiglu", out_fmt="e4m3", want_col=True,
                      pad_to=32, seed=6)
    out = oracle_run(p)
    d = out["d_ref"]
    q = torch.from_numpy(out["d"].reshape(p.m_pad, -1).copy()).view(torch.float8_e4m3fn).double().numpy()
    kb = (2 * p.n) // 32
    for r in range(0, p.m_pad, 7):
        for blk in range(kb):
            code = out["sfd_row"][orc.sf_offset(r, blk, 0, p.m_pad, kb)]
            am = np.abs(d[r, 32 * blk:32 * blk + 32]).max()
            sfd = 2.0 ** (int(code) - 127)
            if am == 0:
                assert code == 0
                continue
            assert sfd >= am / 448 * (1 - 1e-7) and sfd / 2 < am / 448
            deq = q[r, 32 * blk:32 * blk + 32] * sfd
            assert np.all(np.abs(deq - d[r, 32 * blk:32 * blk + 32]) <= am * 2.0 ** -3 + 1e-30)


@pytest.mark.parametrize("epi", ["dswiglu", "dgeglu", "dsituglu"])
def test_dbias_is_the_row_sum_of_d_per_group(epi):
    # every row of every group listed: dbias[g] is numpy's sum of the oracle's
    # D over the group's padded rows (padding rows contribute 0)
    p = small_problem(counts=(40, 0, 70, 33), k=64, n=96, epi=epi, out_fmt="f32", pad_to=32, seed=12)
    out = oracle_run(p)
    off = np_(p.padded_offsets)
    start = 0
    for g in range(p.num_groups):
        want = out["d_ref"][start:int(off[g])].sum(axis=0) if off[g] > start else np.zeros(2 * p.n)
        np.testing.assert_allclose(out["dbias"][g], want, rtol=1e-12, atol=1e-12 * np.abs(want).max(initial=1.0))
        start = int(off[g])
