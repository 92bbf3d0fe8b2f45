"""Pins for the forward epilogue variants of "Grouped GEMM + GLU + Hadamard +
Quant (SM100)", Equations, in the oracle:

* C = alpha_g * sum_k ... + bias_g[n]: the oracle's c_ref against the brute-force
  dense matmul plus the bias, and D computed from it;
* GeGLU: D = gamma * prob * (U + 1) * G * sigmoid(1.702 G), against brute force
  and at closed-form points (G = 0, U = -1, sigmoid = 3/4);
* glu_limit clamps both halves to [-limit, limit] before the activation;
  glu_alpha scales the GLU output; neither touches sReLU;
* c_ref is the value before any clamp or activation.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from helpers import brute_force_C, np_, oracle_run, small_problem

GELU_K = 1.702


def _e4m3(x):
    return int(torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def _single_term(b_codes, alpha=1.0, prob=1.0, a_code=0x38, epi="geglu", m=32):
    """K = 32 with only k = 0 non-zero and unit scales: C[m, n] = alpha * a * b_n."""
    n = len(b_codes)
    p = small_problem(counts=(m,), k=32, n=n, epi=epi, out_fmt="f32", pad_to=32)
    a = torch.zeros(m, 32, dtype=torch.uint8)
    a[:, 0] = a_code
    b = torch.zeros(1, n, 32, dtype=torch.uint8)
    b[0, :, 0] = torch.tensor(b_codes, dtype=torch.uint8)
    p.a, p.b = a, b
    p.sfa_rows = torch.full_like(p.sfa_rows, 127)
    p.sfb_rows = torch.full_like(p.sfb_rows, 127)
    p.alpha = torch.tensor([alpha], dtype=torch.float32)
    p.prob = torch.full((m,), prob, dtype=torch.float32)
    return p


def _bias(p, seed=3):
    g = np.random.default_rng(seed)
    return g.normal(0.0, 2.0, size=(p.num_groups, p.n)).astype(np.float32)


def _rows(p):
    return np.arange(p.m_pad) < np_(p.padded_offsets)[-1]


def _C_with_bias(p, bias):
    C = brute_force_C(p)
    off = np_(p.padded_offsets)
    start = 0
    for g in range(p.num_groups):
        C[start:off[g]] += bias[g].astype(np.float64)
        start = int(off[g])
    return C


@pytest.mark.parametrize("epi", ["gate", "swiglu", "srelu", "geglu"])
def test_c_ref_is_gemm_plus_bias(epi):
    p = small_problem(epi=epi, n=128, k=64, seed=60)
    bias = _bias(p)
    res = oracle_run(p, bias=bias, want_c=True)
    want = _C_with_bias(p, bias)
    rows = _rows(p)
    np.testing.assert_allclose(res["c_ref"][rows], want[rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gate_first", [0, 1])
def test_geglu_matches_brute_force_with_bias(gate_first):
    p = small_problem(epi="geglu", n=128, k=64, seed=61)
    bias = _bias(p, seed=4)
    res = oracle_run(p, bias=bias, gate_first=gate_first)
    Cb = _C_with_bias(p, bias).reshape(p.m_pad, p.n // 64, 2, 32)
    U, G = (Cb[:, :, 1, :], Cb[:, :, 0, :]) if gate_first else (Cb[:, :, 0, :], Cb[:, :, 1, :])
    want = np_(p.prob)[:, None] * ((U + 1.0) * G * expit(GELU_K * G)).reshape(p.m_pad, p.n // 2)
    rows = _rows(p)
    np.testing.assert_allclose(res["d_ref"][rows], want[rows], rtol=1e-12, atol=1e-300)


def test_geglu_closed_forms():
    # [U0 | G0 | U1 | G1]: G0 = 0 -> D = 0; U1 = -1 -> D = 0
    codes = [_e4m3(3.0)] * 32 + [0] * 32 + [_e4m3(-1.0)] * 32 + [_e4m3(2.0)] * 32
    d = oracle_run(_single_term(codes, prob=0.5))["d_ref"][0]
    assert (d == 0.0).all()
    # G = ln 3 / 1.702 makes sigmoid(1.702 G) = 3/4: D = prob * (U + 1) * G * 3/4
    g = float(np.float32(math.log(3.0) / GELU_K))
    p = _single_term([_e4m3(1.0)] * 64, prob=0.25, alpha=g)   # U = G = g
    d = oracle_run(p)["d_ref"][0]
    assert np.allclose(d, 0.25 * (g + 1.0) * g * 0.75, rtol=1e-6)


@pytest.mark.parametrize("epi", ["swiglu", "geglu"])
def test_glu_limit_clamps_both_halves_before_the_activation(epi):
    # X/U = 6, G = 5 (first pair); X/U = -4, G = -3 (second pair); limit 2
    codes = [_e4m3(6.0)] * 32 + [_e4m3(5.0)] * 32 + [_e4m3(-4.0)] * 32 + [_e4m3(-3.0)] * 32
    p = _single_term(codes, epi=epi, prob=0.5)
    res = oracle_run(p, glu_limit=2.0, want_c=True)
    d = res["d_ref"][0]
    if epi == "swiglu":
        f = lambda u, g: u * g * expit(g)
    else:
        f = lambda u, g: (u + 1.0) * g * expit(GELU_K * g)
    assert np.allclose(d[:32], 0.5 * f(2.0, 2.0), rtol=1e-15)
    assert np.allclose(d[32:], 0.5 * f(-2.0, -2.0), rtol=1e-15)
    # C is stored before the clamp
    assert (res["c_ref"][0, :32] == 6.0).all() and (res["c_ref"][0, 32:64] == 5.0).all()
    # within the limit nothing changes
    same = oracle_run(p, glu_limit=100.0)["d_ref"][0]
    base = oracle_run(p)["d_ref"][0]
    assert (same == base).all()


@pytest.mark.parametrize("epi", ["swiglu", "geglu"])
def test_glu_alpha_scales_the_output(epi):
    p = small_problem(epi=epi, n=128, k=64, seed=62)
    base = oracle_run(p)["d_ref"]
    scaled = oracle_run(p, glu_alpha=1.5)["d_ref"]
    np.testing.assert_allclose(scaled, 1.5 * base, rtol=1e-15, atol=0)


def test_glu_options_do_not_touch_srelu_or_gate():
    for epi in ("srelu", "gate"):
        p = small_problem(epi=epi, n=64, k=64, seed=63)
        base = oracle_run(p)["d_ref"]
        other = oracle_run(p, glu_limit=0.5, glu_alpha=3.0)["d_ref"]
        assert (base == other).all()
