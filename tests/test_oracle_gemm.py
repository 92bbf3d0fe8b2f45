"""Pins for the oracle's GEMM, epilogue and output quantization.

* brute force: an independent dense dequantization (torch float8 decoding, the
  listed E2M1 values) and a textbook per-group matmul;
* closed forms of SwiGLU, sReLU and the tanh soft clamp at chosen points;
* invariants: zero prob, linearity in alpha, expert permutation, padding rows,
  empty groups;
* the hand-worked examples in tests/golden/hand_example.json (MXFP8) and
  tests/golden/hand_example_nvfp4.json (NVFP4);
* defining properties of the block quantizer (scale is the power of two at or
  above norm*amax/q_max; dequantized values within one output step of D).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle as orc
from helpers import (E2M1_VALUES, brute_force_C, np_, oracle_inputs, oracle_run, small_problem)
from block_scaled_grouped_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _randomize_scales(p, seed=5):
    """Spread the scale codes so that a wrong scale index changes the result."""
    g = torch.Generator().manual_seed(seed)
    if p.in_fmt == "nvfp4":
        lo, hi = 0x28, 0x48          # E4M3 scales 0.125 .. 2.0
    else:
        lo, hi = 118, 136            # UE8M0 scales 2^-9 .. 2^9
    p.sfa_rows = torch.randint(lo, hi, p.sfa_rows.shape, generator=g).to(torch.uint8)
    p.sfb_rows = torch.randint(lo, hi, p.sfb_rows.shape, generator=g).to(torch.uint8)
    return p


def _rows_in_groups(p):
    off = np_(p.padded_offsets)
    return np.arange(p.m_pad) < off[-1]


@pytest.mark.parametrize("in_fmt", ["mxfp8_e4m3", "mxfp8_e5m2", "nvfp4"])
def test_gate_matches_brute_force(in_fmt):
    p = _randomize_scales(small_problem(in_fmt=in_fmt, k=160, n=96))
    res = oracle_run(p, threads=4)
    C = brute_force_C(p)
    want = np_(p.prob)[:, None].astype(np.float64) * C
    rows = _rows_in_groups(p)
    np.testing.assert_allclose(res["d_ref"][rows], want[rows], rtol=1e-12, atol=0)


def test_1024_groups_mostly_empty_match_brute_force():
    """The largest group count the pages allow (L = 1024), with a few
    non-empty groups scattered among empty ones, some at either end: every
    row takes its own expert's B, scales and alpha; per-group amax is the
    maximum over the group's rows, 0 for an empty group."""
    counts = np.zeros(1024, dtype=np.int64)
    rng = np.random.default_rng(9)
    for g in [0, 1, 517, 518, 900, 1023] + list(rng.choice(np.arange(2, 1023), 6, replace=False)):
        counts[g] = int(rng.integers(1, 70))
    p = _randomize_scales(small_problem(counts=tuple(int(c) for c in counts), k=64, n=64, seed=90))
    res = oracle_run(p)
    C = brute_force_C(p)
    want = np_(p.prob)[:, None].astype(np.float64) * C
    rows = _rows_in_groups(p)
    np.testing.assert_allclose(res["d_ref"][rows], want[rows], rtol=1e-12, atol=0)
    off = np_(p.padded_offsets)
    start = 0
    for g in range(1024):
        blk = res["d_ref"][start:int(off[g])]
        assert res["amax"][g] == (np.float32(np.abs(blk).astype(np.float32).max()) if blk.size else 0.0)
        start = int(off[g])


def test_nonsquare_operands_are_not_transposed():
    p = _randomize_scales(small_problem(counts=(40, 24), k=64, n=160))
    res = oracle_run(p)
    C = brute_force_C(p)
    np.testing.assert_allclose(res["d_ref"], np_(p.prob)[:, None] * C, rtol=1e-12)


def test_swiglu_matches_brute_force():
    p = _randomize_scales(small_problem(epi="swiglu", n=128, k=64))
    res = oracle_run(p)
    C = brute_force_C(p)
    # pair 32-column blocks: [X0 | G0 | X1 | G1 | ...]
    Cb = C.reshape(p.m_pad, p.n // 64, 2, 32)
    X, G = Cb[:, :, 0, :], Cb[:, :, 1, :]
    want = np_(p.prob)[:, None] * (X * G * expit(G)).reshape(p.m_pad, p.n // 2)
    rows = _rows_in_groups(p)
    np.testing.assert_allclose(res["d_ref"][rows], want[rows], rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("s", [0.0, 8.0])
def test_srelu_matches_brute_force(s):
    p = _randomize_scales(small_problem(epi="srelu", n=64, k=64, tanh_clamp_s=s))
    res = oracle_run(p)
    C = brute_force_C(p)
    r = np.maximum(C, 0.0)
    if s:
        r = s * np.tanh(r / s)
    want = np_(p.prob)[:, None] * r * r
    rows = _rows_in_groups(p)
    np.testing.assert_allclose(res["d_ref"][rows], want[rows], rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------------------
# hand-built single-term problems: C[m, n] = alpha * a_m * b_n exactly
# ---------------------------------------------------------------------------

def _single_term(b_codes, alpha=1.0, prob=1.0, a_code=0x38, epi="gate", out_fmt="f32",
                 s=0.0, norm=1.0, want_col=False, m=32):
    """K = 32 with only k = 0 non-zero; unit scales."""
    n = len(b_codes)
    p = small_problem(counts=(m,), k=32, n=n, epi=epi, out_fmt=out_fmt, pad_to=32,
                      tanh_clamp_s=s, norm_const=norm, want_col=want_col)
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


def _e4m3(x):
    return int(torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def test_unit_scales_reproduce_exact_fp8_products():
    vals = [0.5, -1.5, 448.0, 2.0 ** -9, -0.0, 3.0]
    codes = [_e4m3(v) for v in vals]
    p = _single_term(codes, a_code=_e4m3(-6.0), out_fmt="f32")
    d = oracle_run(p)["d_ref"][0]
    assert list(d) == [-6.0 * v for v in vals]


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    m, n, k = g["m"], g["n"], g["k"]
    p = small_problem(counts=(m,), k=k, n=n, out_fmt="e4m3", pad_to=32, want_col=True,
                      norm_const=g["norm_const"])
    p.a = torch.full((m, k), g["a_code"], dtype=torch.uint8)
    p.b = torch.full((1, n, k), g["b_code"], dtype=torch.uint8)
    p.sfa_rows = torch.full_like(p.sfa_rows, g["sf_code"])
    p.sfb_rows = torch.full_like(p.sfb_rows, g["sf_code"])
    p.alpha = torch.tensor([g["alpha"]])
    p.prob = torch.full((m,), g["prob"])
    res = oracle_run(p)
    e = g["expected"]
    assert (res["d_ref"] == e["D"]).all()
    assert (res["d"] == e["dq_code"]).all() and (res["d_col"] == e["dq_code"]).all()
    assert (res["sfd_row"][:orc.sf_bytes(m, 1, 1)].reshape(-1)[
        [orc.sf_offset(r, 0, 0, m, 1) for r in range(m)]] == e["sfd_code"]).all()
    assert (res["sfd_col"][[orc.sf_offset(c, 0, 0, n, 1) for c in range(n)]] == e["sfd_code"]).all()


def test_hand_worked_nvfp4_example():
    """tests/golden/hand_example_nvfp4.json: E2M1 data with E4M3 scales per 16
    (two K blocks holding different values and scales), E2M1 output with
    E4M3 row scales, 16-row column blocks and a round-to-nearest-even tie."""
    g = json.load(open(os.path.join(GOLDEN, "hand_example_nvfp4.json")))
    m, n, k = g["m"], g["n"], g["k"]
    p = small_problem(counts=(m,), k=k, n=n, in_fmt="nvfp4", out_fmt="e2m1", pad_to=32,
                      want_col=True, norm_const=g["norm_const"])
    nib_a = np.repeat(np.array(g["a_codes_by_kblock"], dtype=np.uint8), 16)          # (k,)
    a = nib_a[0::2] | (nib_a[1::2] << 4)
    p.a = torch.from_numpy(np.tile(a, (m, 1)))
    p.sfa_rows = torch.from_numpy(np.tile(np.array(g["sfa_by_kblock"], dtype=np.uint8), (1, m, 1)))
    b_codes = np.concatenate([np.tile(np.array(blk, dtype=np.uint8), 4) for blk in g["b_pattern"]])  # (n,)
    p.b = torch.from_numpy(np.repeat((b_codes | (b_codes << 4))[None, :, None], k // 2, axis=2))
    p.sfb_rows = torch.full((1, n, k // 16), g["sfb_code"], dtype=torch.uint8)
    p.alpha = torch.tensor([g["alpha"]])
    p.prob = torch.full((m,), g["prob"])
    res = oracle_run(p)
    e = g["expected"]
    per_col = lambda key: np.concatenate([np.tile(np.array(blk), 4) for blk in e[key]])
    assert (res["d_ref"] == per_col("d_by_block")[None, :]).all()
    unpack = lambda raw: np.stack([raw & 0xF, raw >> 4], axis=-1).reshape(m, n)
    assert (unpack(res["d"].reshape(m, n // 2)) == per_col("dq_codes_by_block")[None, :]).all()
    assert (unpack(res["d_col"].reshape(m, n // 2)) == per_col("dcol_codes_by_block")[None, :]).all()
    for r in range(m):
        for b in range(n // 16):
            assert res["sfd_row"][orc.sf_offset(r, b, 0, m, n // 16)] == e["sfd_row_codes"][b]
    sfd_col = per_col("sfd_col_codes_by_block")
    for c in range(n):
        for b in range(m // 16):
            assert res["sfd_col"][orc.sf_offset(c, b, 0, n, m // 16)] == sfd_col[c]


def test_swiglu_closed_forms_and_block_pairing():
    # columns [0,32) = X0 = 1, [32,64) = G0 = 8, [64,96) = X1 = 4, [96,128) = G1 = 0
    codes = [_e4m3(1.0)] * 32 + [_e4m3(8.0)] * 32 + [_e4m3(4.0)] * 32 + [0] * 32
    p = _single_term(codes, epi="swiglu", prob=0.5)
    d = oracle_run(p)["d_ref"][0]
    sig8 = 1.0 / (1.0 + math.exp(-8.0))
    assert np.allclose(d[:32], 0.5 * 1.0 * 8.0 * sig8, rtol=1e-15)
    assert (d[32:] == 0.0).all()                      # swish(0) = 0
    # G = ln 3: sigmoid(ln 3) = 3/4, so D = prob * X * ln3 * 3/4
    ln3 = float(np.float32(math.log(3.0)))
    p = _single_term([_e4m3(1.0)] * 64, epi="swiglu", prob=0.25, alpha=ln3)
    d = oracle_run(p)["d_ref"][0]
    assert np.allclose(d, 0.25 * ln3 * ln3 * 0.75, rtol=1e-7)


def test_swiglu_gate_first_order_is_one_switch_away():
    codes = [_e4m3(1.0)] * 32 + [_e4m3(8.0)] * 32
    p = _single_term(codes, epi="swiglu")
    d_first = oracle_run(p, gate_first=1)["d_ref"][0]
    sig1 = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(d_first, 8.0 * 1.0 * sig1, rtol=1e-15)


def test_srelu_closed_forms():
    p = _single_term([_e4m3(2.0), _e4m3(-2.0), 0], epi="srelu", prob=0.75)
    d = oracle_run(p)["d_ref"][0]
    assert list(d) == [0.75 * 4.0, 0.0, 0.0]
    s = 8.0
    c = float(np.float32(s * math.atanh(0.5)))     # tanh(c/s) = 1/2 -> D = prob*s^2/4
    p = _single_term([_e4m3(1.0)], epi="srelu", prob=0.5, alpha=c, s=s)
    d = oracle_run(p)["d_ref"][0]
    assert np.allclose(d, 0.5 * s * s / 4.0, rtol=1e-6)
    # soft clamp bounds D by prob * s^2 ("Grouped GEMM + sReLU", Tanh soft clamp)
    p = _single_term([_e4m3(448.0)], epi="srelu", prob=0.5, alpha=64.0, s=s)
    d = oracle_run(p)["d_ref"][0]
    assert d[0] <= 0.5 * s * s and d[0] > 0.5 * s * s * (1 - 1e-12)
    assert orc.srelu(-3.0, 0.0) == 0.0 and orc.srelu(3.0, 0.0) == 9.0
    assert orc.sigmoid(0.0) == 0.5


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_zero_prob_rows_are_zero_and_quantize_to_zero():
    p = small_problem(out_fmt="e4m3", want_col=True, n=64)
    prob = np_(p.prob).copy()
    prob[:32] = 0.0
    res = oracle_run(p, prob=prob)
    assert (res["d_ref"][:32] == 0.0).all()
    assert ((res["d"][:32] & 0x7F) == 0).all()
    kb = p.n_out // 32
    for r in range(32):
        for j in range(kb):
            assert res["sfd_row"][orc.sf_offset(r, j, 0, p.m_pad, kb)] == 0


def test_linear_in_alpha():
    p = _randomize_scales(small_problem())
    base = oracle_run(p)["d_ref"]
    doubled = oracle_run(p, alpha=np_(p.alpha) * 2.0)["d_ref"]
    assert np.array_equal(doubled, 2.0 * base)


def test_padding_rows_are_zero_and_empty_groups_have_zero_amax():
    p = small_problem(counts=(70, 0, 130, 20), pad_to=32)
    res = oracle_run(p)
    off = np_(p.padded_offsets)
    starts = np.concatenate([[0], off[:-1]])
    for g, c in enumerate(p.counts):
        assert (res["d_ref"][starts[g] + c:off[g]] == 0.0).all()
    assert res["amax"][1] == 0.0
    assert all(res["amax"][g] > 0 for g in (0, 2, 3))
    # amax is the max |D| over the group's rows
    for g in (0, 2, 3):
        blk = res["d_ref"][starts[g]:off[g]]
        assert res["amax"][g] == np.float32(np.abs(blk).max())


def test_expert_permutation_permutes_rows():
    counts = (64, 32, 96)
    p = _randomize_scales(small_problem(counts=counts, pad_to=32))
    ins = oracle_inputs(p)
    base = oracle_run(p, inputs=ins)["d_ref"]
    perm = [2, 0, 1]
    off = np_(p.padded_offsets)
    starts = np.concatenate([[0], off[:-1]])
    rows = np.concatenate([np.arange(starts[g], off[g]) for g in perm])
    sfa_rows = np_(p.sfa_rows)[:, rows]
    new = dict(ins)
    new["a"] = ins["a"][rows]
    new["sfa"] = orc.pack_sf(sfa_rows)
    new["b"] = ins["b"][perm]
    new["sfb"] = orc.pack_sf(np_(p.sfb_rows)[perm])
    new["alpha"] = ins["alpha"][perm]
    new["prob"] = ins["prob"][rows]
    new["padded_offsets"] = np.cumsum([off[g] - starts[g] for g in perm]).astype(np.int32)
    got = oracle_run(p, inputs=new)["d_ref"]
    assert np.array_equal(got, base[rows])


def test_rows_after_last_offset_are_untouched():
    p = small_problem(counts=(64,), pad_to=32, out_fmt="e4m3")
    ins = oracle_inputs(p)
    res = orc.run(m_pad=96, n=p.n, k=p.k, num_groups=1, in_fmt=orc.IN_MXFP8_E4M3,
                  out_fmt=orc.OUT_E4M3, epi=orc.EPI_GATE,
                  a=np.concatenate([ins["a"], np.zeros((32, p.k), np.uint8)]),
                  sfa=orc.pack_sf(np.concatenate([np_(p.sfa_rows), np.full((1, 32, 3), 127, np.uint8)], 1)),
                  b=ins["b"], sfb=ins["sfb"], padded_offsets=ins["padded_offsets"],
                  alpha=ins["alpha"], prob=np.concatenate([ins["prob"], np.ones(32, np.float32)]),
                  outputs={"d": np.full((96, p.n), 0xAB, np.uint8)})
    assert (res["d"][64:] == 0xAB).all()
    assert (res["d"][:64] != 0xAB).any()


# ---------------------------------------------------------------------------
# quantizer properties
# ---------------------------------------------------------------------------

def _decode_out(codes, fmt):
    if fmt == "e2m1":
        nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
        return E2M1_VALUES[nib]
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes)).view(dt).double().numpy()


def _decode_sf(codes, in_fmt):
    dt = torch.float8_e4m3fn if in_fmt == "nvfp4" else torch.float8_e8m0fnu
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(dt).double().numpy()


def _check_scale(sf, target, in_fmt):
    """The block scale's rounding rule: UE8M0 is the least power of two at or
    above the target; an E4M3 scale is the nearest E4M3 value (half a step is
    2^-4 relative), saturating at 448, and zero below half the smallest
    subnormal 2^-9.  Returns "ok", "saturated" (the data saturate too) or
    "zero" (the block is written as zeros)."""
    if in_fmt != "nvfp4":
        assert sf >= target * (1 - 1e-6) and sf / 2 < target * (1 + 1e-6)
        return "ok"
    if target >= 448.0:
        assert sf == 448.0
        return "saturated"
    if sf == 0.0:
        assert target <= 2.0 ** -10
        return "zero"
    assert abs(sf - target) <= target * 2 ** -4 + 2 ** -10
    return "ok"


# Signed D (gating) and non-negative D (sReLU); more than one 128-row tile of
# the scale layout (m_pad 224), column blocks of 32 and of 16 rows.
@pytest.mark.parametrize("in_fmt,out_fmt,norm,epi", [("mxfp8_e4m3", "e4m3", 1.0, "srelu"),
                                                     ("mxfp8_e4m3", "e4m3", 1.0, "gate"),
                                                     ("mxfp8_e4m3", "e5m2", 0.5, "srelu"),
                                                     ("mxfp8_e5m2", "e4m3", 2.0, "gate"),
                                                     ("mxfp8_e4m3", "e2m1", 1.0, "srelu"),
                                                     ("nvfp4", "e2m1", 1.0, "srelu"),
                                                     ("nvfp4", "e2m1", 1.0, "gate"),
                                                     ("nvfp4", "e2m1", 2.0 ** -12, "srelu"),
                                                     ("fp4_ue8m0_16", "e2m1", 1.0, "gate")])
def test_row_and_column_quantization_properties(in_fmt, out_fmt, norm, epi):
    p = _randomize_scales(small_problem(in_fmt=in_fmt, out_fmt=out_fmt, epi=epi,
                                        n=128, k=64, counts=(100, 90), pad_to=32,
                                        norm_const=norm, want_col=1))
    assert p.m_pad > 128
    res = oracle_run(p)
    v = p.sf_vec
    qmax = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}[out_fmt]
    step = {"e4m3": 2 ** -3, "e5m2": 2 ** -2, "e2m1": 1.0 / 3.0}[out_fmt]
    D = res["d_ref"].astype(np.float32).astype(np.float64)
    if epi == "gate":
        assert (D < 0).any()
    nd = p.n_out
    rows = _rows_in_groups(p)
    # row blocks
    Dq = _decode_out(res["d"], out_fmt)
    sf_row = np.array([[res["sfd_row"][orc.sf_offset(r, j, 0, p.m_pad, nd // v)]
                        for j in range(nd // v)] for r in range(p.m_pad)])
    sfd = _decode_sf(sf_row, in_fmt)
    for r in np.nonzero(rows)[0]:
        for j in range(nd // v):
            blk = D[r, j * v:(j + 1) * v]
            am = np.abs(blk).max()
            if am == 0:
                continue
            kind = _check_scale(sfd[r, j], norm * am / qmax, in_fmt)
            if kind == "zero":
                assert np.all(Dq[r, j * v:(j + 1) * v] == 0)
            if kind != "ok":
                continue
            deq = Dq[r, j * v:(j + 1) * v] * sfd[r, j] / norm
            # within one output step of the block's scale (coarsest step at the top)
            assert np.all(np.abs(deq - blk) <= step * am + 1e-30)
    # column blocks of v rows, SFD_col in SF(n_d, m_pad)
    Dc = _decode_out(res["d_col"], out_fmt)
    for j in range(nd):
        for b in range(p.m_pad // v):
            blk_rows = np.arange(b * v, b * v + v)
            blk_rows = blk_rows[rows[blk_rows]]
            if blk_rows.size == 0:
                continue
            am = np.abs(D[blk_rows, j]).max()
            sf = _decode_sf(np.array([res["sfd_col"][orc.sf_offset(j, b, 0, nd, p.m_pad // v)]]),
                            in_fmt)[0]
            if am == 0:
                continue
            kind = _check_scale(sf, norm * am / qmax, in_fmt)
            if kind == "zero":
                assert np.all(Dc[blk_rows, j] == 0)
            if kind != "ok":
                continue
            deq = Dc[blk_rows, j] * sf / norm
            assert np.all(np.abs(deq - D[blk_rows, j]) <= step * am + 1e-30)


@pytest.mark.parametrize("in_fmt", ["fp4_ue8m0_16", "mxfp4"])
def test_fp4_with_ue8m0_scales_against_brute_force(in_fmt):
    """FP4 data with UE8M0 scales per 16 or per 32 ("Grouped GEMM + Quant
    (SM100)", Data Types: NVF4 with float8_e8m0fnu scales): C against the
    brute-force dense matmul (torch's e8m0 decoding, E2M1 listed values), with
    spread scales; quantized E2M1 output with UE8M0 block scales rounded up."""
    from helpers import brute_force_C, oracle_run, small_problem, np_
    p = small_problem(counts=(40, 0, 70), k=192, n=64, in_fmt=in_fmt, out_fmt="f32", seed=17)
    g = torch.Generator().manual_seed(4)
    p.sfa_rows = torch.randint(120, 134, p.sfa_rows.shape, generator=g).to(torch.uint8)
    p.sfb_rows = torch.randint(120, 134, p.sfb_rows.shape, generator=g).to(torch.uint8)
    out = oracle_run(p)
    C = brute_force_C(p)
    rows = ~np.isnan(C[:, 0])
    want = C * np_(p.prob)[:, None]
    np.testing.assert_allclose(out["d_ref"][rows], want[rows], rtol=1e-12, atol=1e-9)
    # E2M1 output: per 16 (or 32) columns a UE8M0 scale = least power of two >= max|D| / 6
    q = small_problem(counts=(64,), k=128, n=64, in_fmt=in_fmt, out_fmt="e2m1", seed=18)
    oq = oracle_run(q)
    v = 32 if in_fmt == "mxfp4" else 16
    import oracle as orc
    for r in range(0, 64, 9):
        for b in range(64 // v):
            code = int(oq["sfd_row"][orc.sf_offset(r, b, 0, q.m_pad, 64 // v)])
            am = float(np.abs(oq["d_ref"][r, v * b:v * b + v]).astype(np.float32).max())
            if am == 0:
                assert code == 0
                continue
            sf = 2.0 ** (code - 127)
            assert sf >= am / 6 * (1 - 1e-6) and sf / 2 < am / 6
