"""Pins for the oracle's bfloat16 operands: the BF16 backend of "Grouped GEMM +
dGLU (SM100)" (BF16 contract: bfloat16 A and B, no scale factors,
R_g = alpha_g^2 A_g B_g^T, X_g = beta_g C_g).

* the GEMM step on bfloat16 operands against the brute-force dense matmul
  (torch's bfloat16 decoding of the little-endian byte pairs);
* the backward epilogues do not depend on the input family: MXFP8 E4M3 codes
  with unit scales, rewritten as the same values in bfloat16 (every finite
  E4M3 value is a bfloat16 value), give bit-identical dSwiGLU and dSiTU-GLU
  outputs and dprob;
* dGeGLU reads beta on bfloat16 operands and only there: with beta = 2 the
  BF16 result equals the MXFP8 result on a saved C doubled (exact), while the
  block-scaled result ignores beta.
"""
import numpy as np
import pytest
import torch

from helpers import brute_force_C, np_, oracle_run, small_problem


def test_bf16_gemm_against_brute_force():
    p = small_problem(counts=(40, 0, 70, 9), k=200, n=96, in_fmt="bf16", out_fmt="f32", seed=31)
    assert p.a.shape == (p.m_pad, 2 * p.k) and p.sfa_rows.shape[-1] == 0
    out = oracle_run(p)
    C = brute_force_C(p)
    rows = ~np.isnan(C[:, 0])
    want = C * np_(p.prob)[:, None]
    np.testing.assert_allclose(out["d_ref"][rows], want[rows], rtol=1e-12, atol=1e-12)
    # bfloat16 values of the generator: the RNE of the float32 draws
    x = torch.from_numpy(np_(p.a)).view(torch.bfloat16).float()
    assert torch.all(torch.isfinite(x)) and x.abs().max() > 0


def _as_bf16_problem(p):
    """The same values as MXFP8 problem p (unit scales) in bfloat16 bytes."""
    q = small_problem(counts=tuple(int(c) for c in p.counts), k=p.k, n=p.n, in_fmt="bf16",
                      out_fmt=p.out_fmt, epi=p.epi, pad_to=32, seed=1)
    a = torch.from_numpy(np_(p.a)).view(torch.float8_e4m3fn).float().to(torch.bfloat16)
    b = torch.from_numpy(np_(p.b)).view(torch.float8_e4m3fn).float().to(torch.bfloat16)
    assert torch.equal(a.float(), torch.from_numpy(np_(p.a)).view(torch.float8_e4m3fn).float())
    q.a = a.contiguous().view(torch.uint8).reshape(p.m_pad, 2 * p.k)
    q.b = b.contiguous().view(torch.uint8).reshape(p.num_groups, p.n, 2 * p.k)
    q.padded_offsets, q.alpha, q.prob = p.padded_offsets, p.alpha, p.prob
    q.saved_c, q.beta = p.saved_c, p.beta
    return q


def _unit_scale_mxfp8(epi, seed):
    p = small_problem(counts=(45, 0, 64), k=128, n=64, in_fmt="mxfp8_e4m3", out_fmt="f32", epi=epi,
                      pad_to=32, seed=seed)
    p.sfa_rows = torch.full_like(p.sfa_rows, 127)
    p.sfb_rows = torch.full_like(p.sfb_rows, 127)
    return p


@pytest.mark.parametrize("epi", ["dswiglu", "dsituglu"])
def test_backward_epilogue_independent_of_input_family(epi):
    p = _unit_scale_mxfp8(epi, seed=41)
    q = _as_bf16_problem(p)
    # one thread: dprob and dbias then sum their column slices in one order
    o8, o16 = oracle_run(p, threads=1), oracle_run(q, threads=1)
    assert np.array_equal(o8["d_ref"], o16["d_ref"])
    assert np.array_equal(o8["dprob_ref"], o16["dprob_ref"])
    assert np.array_equal(o8["dbias"], o16["dbias"])
    assert np.abs(o8["d_ref"]).max() > 0


def test_dgeglu_reads_beta_on_bf16_only():
    p = _unit_scale_mxfp8("dgeglu", seed=43)
    p.beta = torch.full_like(p.beta, 2.0)
    q = _as_bf16_problem(p)
    o8 = oracle_run(p, threads=1)
    o16 = oracle_run(q, threads=1)
    # block-scaled: beta ignored (the same as beta = 1)
    p1 = _unit_scale_mxfp8("dgeglu", seed=43)
    p1.beta = torch.ones_like(p1.beta)
    assert np.array_equal(o8["d_ref"], oracle_run(p1)["d_ref"])
    # BF16: X = beta C, i.e. the block-scaled result on 2 C
    doubled = oracle_run(p, saved_c=np_(p.saved_c.double()) * 2.0, threads=1)
    assert np.array_equal(o16["d_ref"], doubled["d_ref"])
    assert np.array_equal(o16["dprob_ref"], doubled["dprob_ref"])
    assert not np.array_equal(o16["d_ref"], o8["d_ref"])
