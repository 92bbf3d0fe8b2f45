"""Pins for the oracle's dGeGLU backward ("Grouped GEMM + dGLU (SM100)",
Block-scaled contract, Step 2, dGeGLU):

* inside the clamp range, the gradients are ref * d(forward GeGLU)/d(up, gate):
  central finite differences of the oracle's own forward GeGLU (pinned
  separately), evaluated at chosen points through the bias (A = 0);
* dprob is the sum of ref * (forward GeGLU at unit prob) inside the range;
* clamps and masks at closed-form points: the gate has only an upper clamp,
  the up value both; a value beyond a bound zeroes its own gradient and enters
  the other one clamped; a value at a bound keeps its gradient;
* geglu_alpha = 1 and linear_offset = 0 make dGeGLU the dSwiGLU of the same
  saved C (beta = 1), itself pinned by finite differences;
* beta is not read.

And for the dSiTU-GLU backward (same page, Equations): the gradients against
central finite differences of the page's defining product T_g * T_u
(T_g = b1 tanh(G/b1) sigmoid(G), T_u = b2 tanh(U/b2)) for several b1, b2, dprob
against ref * T_g * T_u, and closed forms at G = 0 and U = 0.
"""
import numpy as np
import pytest
import torch

from helpers import oracle_run, small_problem

POINTS = [(0.5, 1.5), (-2.0, 0.75), (3.0, -1.25), (-0.25, -3.0), (1.5, 4.0), (6.5, -6.0)]


def _forward_geglu(pairs, prob=1.0, h=0.0, which=None):
    """Forward GeGLU D of the oracle at (up, gate) points, C = bias (A = 0), no
    clamp.  Block order [up | gate] (gate_first = 0)."""
    P = len(pairs)
    n = 64 * P
    p = small_problem(counts=(32,), k=32, n=n, epi="geglu", out_fmt="f32", pad_to=32, seed=1)
    p.a = torch.zeros_like(p.a)
    p.alpha = torch.ones(1)
    p.prob = torch.full((32,), prob, dtype=torch.float32)
    bias = np.zeros((1, n))
    for b, (u, g) in enumerate(pairs):
        bias[0, 64 * b:64 * b + 32] = u + (h if which == "u" else 0.0)
        bias[0, 64 * b + 32:64 * b + 64] = g + (h if which == "g" else 0.0)
    return oracle_run(p, bias=bias.astype(np.float32))["d_ref"][0].reshape(P, 32)[:, 0]


def _backward(points, ref_codes, prob=0.75, epi="dgeglu", gate_first=0, beta=1.0, **params):
    P = len(points)
    n = 32 * P
    p = small_problem(counts=(32,), k=32, n=n, epi=epi, out_fmt="f32", pad_to=32, seed=2)
    a = torch.zeros(32, 32, dtype=torch.uint8)
    a[:, 0] = 0x38
    b = torch.zeros(1, n, 32, dtype=torch.uint8)
    b[0, :, 0] = torch.tensor(ref_codes, dtype=torch.uint8).repeat_interleave(32)
    p.a, p.b = a, b
    p.sfa_rows = torch.full_like(p.sfa_rows, 127)
    p.sfb_rows = torch.full_like(p.sfb_rows, 127)
    p.alpha = torch.ones(1)
    p.prob = torch.full((32,), prob, dtype=torch.float32)
    p.beta = torch.tensor([beta], dtype=torch.float32)
    saved = np.zeros((32, 2 * n))
    for blk, (u, g) in enumerate(points):
        uo, go = (64 * blk + 32, 64 * blk) if gate_first else (64 * blk, 64 * blk + 32)
        saved[:, uo:uo + 32] = u
        saved[:, go:go + 32] = g
    p.saved_c = torch.from_numpy(saved).to(torch.bfloat16)
    out = oracle_run(p, gate_first=gate_first, **params)
    d = out["d_ref"][0].reshape(P, 64)
    d_up = d[:, 32] if gate_first else d[:, 0]
    d_gate = d[:, 0] if gate_first else d[:, 32]
    return d_up, d_gate, out


def _bf16(x):
    return float(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double())


REF_CODES = [0x40, 0x38, 0xB8, 0x44, 0x30, 0xC0]    # 2, 1, -1, 3, 0.5, -2
REF = np.array([2.0, 1.0, -1.0, 3.0, 0.5, -2.0])


def test_gradients_inside_the_clamp_range_are_finite_differences_of_the_forward():
    pts = [(_bf16(u), _bf16(g)) for u, g in POINTS]
    d_up, d_gate, _ = _backward(pts, REF_CODES, prob=0.75)
    h = 2.0 ** -12
    dfdu = (_forward_geglu(pts, h=h, which="u") - _forward_geglu(pts, h=-h, which="u")) / (2 * h)
    dfdg = (_forward_geglu(pts, h=h, which="g") - _forward_geglu(pts, h=-h, which="g")) / (2 * h)
    np.testing.assert_allclose(d_up, REF * 0.75 * dfdu, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(d_gate, REF * 0.75 * dfdg, rtol=1e-6, atol=1e-9)


def test_dprob_inside_the_range():
    pts = [(_bf16(u), _bf16(g)) for u, g in POINTS]
    _, _, out = _backward(pts, REF_CODES, prob=0.2)
    want = 32 * np.sum(REF * _forward_geglu(pts, prob=1.0))
    np.testing.assert_allclose(out["dprob_ref"], np.full(32, want), rtol=1e-12)


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


@pytest.mark.parametrize("gate_first", [0, 1])
def test_clamps_and_masks(gate_first):
    # (up, gate): gate beyond the upper bound, gate at it, gate far below (no
    # lower clamp), up above, up below, up at either bound
    pts = [(1.0, 9.0), (1.0, 7.0), (1.0, -9.0), (8.0, 1.0), (-8.0, 1.0), (7.0, 1.0), (-7.0, 2.0)]
    codes = [0x38] * len(pts)                         # ref = 1
    d_up, d_gate, out = _backward(pts, codes, prob=1.0, gate_first=gate_first)
    a, off = 1.702, 1.0
    want_up, want_gate, want_dp = [], [], []
    for u, g in pts:
        gc, uc = min(g, 7.0), min(max(u, -7.0), 7.0)
        s = _sig(a * gc)
        want_gate.append((uc + off) * s * (1 + a * gc * (1 - s)) * (1.0 if g <= 7.0 else 0.0))
        want_up.append(gc * s * (1.0 if -7.0 <= u <= 7.0 else 0.0))
        want_dp.append(gc * s * (uc + off))
    np.testing.assert_allclose(d_up, want_up, rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(d_gate, want_gate, rtol=1e-14, atol=1e-300)
    assert d_gate[0] == 0.0 and d_up[3] == 0.0 and d_up[4] == 0.0      # masked beyond a bound
    assert d_gate[1] != 0.0 and d_up[5] != 0.0 and d_up[6] != 0.0      # kept at a bound
    np.testing.assert_allclose(out["dprob_ref"][0], 32 * np.sum(want_dp), rtol=1e-13)


def test_alpha_one_offset_zero_is_dswiglu():
    rng = np.random.default_rng(3)
    pts = [(_bf16(u), _bf16(g)) for u, g in rng.uniform(-6, 6, size=(6, 2))]
    d_up, d_gate, o1 = _backward(pts, REF_CODES, prob=0.6, geglu_alpha=1.0, linear_offset=0.0,
                                 glu_clamp_min=-10.0, glu_clamp_max=10.0)
    s_up, s_gate, o2 = _backward(pts, REF_CODES, prob=0.6, epi="dswiglu")
    np.testing.assert_allclose(d_up, s_up, rtol=1e-14)
    np.testing.assert_allclose(d_gate, s_gate, rtol=1e-14)
    np.testing.assert_allclose(o1["dprob_ref"], o2["dprob_ref"], rtol=1e-13)


def test_beta_is_not_read():
    pts = [(1.5, 0.5), (-1.0, 2.0)]
    _, _, o1 = _backward(pts, REF_CODES[:2], beta=1.0)
    _, _, o2 = _backward(pts, REF_CODES[:2], beta=3.0)
    assert np.array_equal(o1["d_ref"], o2["d_ref"])
    assert np.array_equal(o1["dprob_ref"], o2["dprob_ref"])


# ---------------------------------------------------------------- dSiTU-GLU
def _situ_forward(u, g, b1, b2):
    """The page's definitions: T_g = b1 tanh(G/b1) sigmoid(G), T_u = b2 tanh(U/b2);
    the gradients returned are those of T_g * T_u."""
    return b1 * np.tanh(g / b1) * _sig(g) * (b2 * np.tanh(u / b2))


@pytest.mark.parametrize("b1,b2", [(1.0, 1.0), (2.0, 0.5), (8.0, 8.0)])
def test_dsitu_gradients_are_finite_differences(b1, b2):
    pts = [(_bf16(u), _bf16(g)) for u, g in POINTS]
    d_up, d_gate, out = _backward(pts, REF_CODES, prob=0.75, epi="dsituglu", situ_beta1=b1, situ_beta2=b2)
    u = np.array([q[0] for q in pts])
    g = np.array([q[1] for q in pts])
    h = 1e-6
    dfdu = (_situ_forward(u + h, g, b1, b2) - _situ_forward(u - h, g, b1, b2)) / (2 * h)
    dfdg = (_situ_forward(u, g + h, b1, b2) - _situ_forward(u, g - h, b1, b2)) / (2 * h)
    np.testing.assert_allclose(d_up, REF * 0.75 * dfdu, rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(d_gate, REF * 0.75 * dfdg, rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(out["dprob_ref"][0], 32 * np.sum(REF * _situ_forward(u, g, b1, b2)), rtol=1e-12)


def test_dsitu_closed_forms():
    # G = 0: T_g = 0, dT_g/dG = 1/2; U = 0: T_u = 0, dT_u/dU = 1
    d_up, d_gate, out = _backward([(0.0, 0.0), (1.0, 0.0), (0.0, 1.0)], [0x40] * 3, prob=0.5, epi="dsituglu",
                                  situ_beta1=2.0, situ_beta2=3.0)
    assert d_up[0] == 0.0 and d_gate[0] == 0.0            # T_u = 0 and T_g = 0
    np.testing.assert_allclose(d_gate[1], 2 * 0.5 * 3.0 * np.tanh(1.0 / 3.0) * 0.5, rtol=1e-15)
    assert d_up[1] == 0.0                                 # T_g = 0 at G = 0
    tg = 2.0 * np.tanh(0.5) * _sig(1.0)
    np.testing.assert_allclose(d_up[2], 2 * 0.5 * tg * 1.0, rtol=1e-15)
    np.testing.assert_allclose(out["dprob_ref"][0], 0.0, atol=0)
