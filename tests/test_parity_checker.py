"""The GPU parity checker itself, on the CPU.

The GPU tests judge the kernel with ``gpu_harness.compare``: BF16/F16/F32 D
within |d - ref| <= 2^-7 |ref| + 1e-3 rms(ref); FP8/FP4 D and their scale
factors bit-equal on >= 99.9 % of codes and blocks and within one code step
elsewhere, a block whose scale is one step off compared by its dequantized
values.  Here the oracle's own outputs stand in for a GPU result, first
unchanged (accepted), then with planted differences that the bar must reject
(two code steps, too many one-step flips, a scale off with its data not
re-quantized, rows of another group, a NaN) or accept (a few one-step flips,
a scale one step off with its block re-quantized consistently, BF16 rounding).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
from gpu_harness import code_rank, compare
from helpers import oracle_run, small_problem


def _problem(out_fmt="e4m3", in_fmt="mxfp8_e4m3"):
    # m_pad 224 (two row tiles of the scale layout), an empty group, signed D;
    # 1792 row and 1792 column scale blocks, so that one differing scale stays
    # under the 0.1 % rate and the step rule decides
    return small_problem(counts=(100, 0, 90), k=64, n=256, pad_to=32, epi="gate",
                         in_fmt=in_fmt, out_fmt=out_fmt, want_col=1, seed=5)


def _outs(ref, keys=("d", "d_col", "sfd_row", "sfd_col")):
    return {k: torch.from_numpy(np.ascontiguousarray(ref[k]).reshape(-1).copy()) for k in keys if k in ref}


@pytest.fixture(scope="module")
def e4m3_case():
    p = _problem()
    return p, oracle_run(p)


def _valid_codes(p, ref, plane="d"):
    """(row, col) of codes in valid rows whose magnitude leaves room for two
    steps up without reaching the NaN code."""
    d = ref[plane].reshape(p.m_pad, -1)
    rows = np.arange(p.m_pad) < int(p.padded_offsets[-1])
    mag = d & 0x7F
    ok = rows[:, None] & (mag >= 0x10) & (mag <= 0x70)
    return np.argwhere(ok)


def _bump(codes, idx, steps):
    """Move E4M3 codes `steps` away from zero (same sign)."""
    c = codes.copy()
    for r, j in idx:
        c[r, j] = np.uint8((int(c[r, j]) & 0x80) | ((int(c[r, j]) & 0x7F) + steps))
    return c


def test_identical_outputs_pass(e4m3_case):
    p, ref = e4m3_case
    compare(p, _outs(ref), ref)


def test_a_code_two_steps_off_fails(e4m3_case):
    p, ref = e4m3_case
    idx = _valid_codes(p, ref)[:1]
    outs = _outs(ref)
    outs["d"] = torch.from_numpy(_bump(ref["d"].reshape(p.m_pad, -1), idx, 2).reshape(-1))
    with pytest.raises(AssertionError, match="steps off"):
        compare(p, outs, ref)


@pytest.mark.parametrize("frac,ok", [(0.0005, True), (0.002, False)])
def test_one_step_flips_pass_only_below_the_rate(e4m3_case, frac, ok):
    p, ref = e4m3_case
    cand = _valid_codes(p, ref)
    n_valid = int(p.padded_offsets[-1]) * p.n_out
    count = max(1, int(frac * n_valid))
    rng = np.random.default_rng(0)
    idx = cand[rng.choice(len(cand), count, replace=False)]
    outs = _outs(ref)
    outs["d"] = torch.from_numpy(_bump(ref["d"].reshape(p.m_pad, -1), idx, 1).reshape(-1))
    if ok:
        compare(p, outs, ref)
    else:
        with pytest.raises(AssertionError, match="of codes equal"):
            compare(p, outs, ref)


def _row_block(p, ref):
    """A valid row and 32-column block whose maximum is well inside E4M3."""
    d_ref = ref["d_ref"]
    r = 3
    am = np.abs(d_ref[r, 0:32]).max()
    assert am > 0
    return r, 0, am


def test_scale_one_step_off_without_requantized_data_fails(e4m3_case):
    p, ref = e4m3_case
    r, b, _ = _row_block(p, ref)
    sf = ref["sfd_row"].copy()
    o = orc.sf_offset(r, b, 0, p.m_pad, p.n_out // 32)
    sf[o] += 1
    outs = _outs(ref)
    outs["sfd_row"] = torch.from_numpy(sf)
    with pytest.raises(AssertionError, match="differing scales"):
        compare(p, outs, ref)


def test_scale_one_step_off_with_requantized_block_passes(e4m3_case):
    """A block quantized under the next power of two: every value re-encoded
    from D with half the scale factor's reciprocal; within one output step."""
    p, ref = e4m3_case
    r, b, _ = _row_block(p, ref)
    sf = ref["sfd_row"].copy()
    o = orc.sf_offset(r, b, 0, p.m_pad, p.n_out // 32)
    sf[o] += 1
    scale = p.norm_const / 2.0 ** (int(sf[o]) - 127)
    d = ref["d"].reshape(p.m_pad, -1).copy()
    for j in range(32 * b, 32 * b + 32):
        d[r, j] = orc.encode_rne_satfinite(orc.F_E4M3, float(np.float32(ref["d_ref"][r, j]) * np.float32(scale)))
    outs = _outs(ref)
    outs["sfd_row"] = torch.from_numpy(sf)
    outs["d"] = torch.from_numpy(d.reshape(-1))
    compare(p, outs, ref)


def test_scale_two_steps_off_fails(e4m3_case):
    p, ref = e4m3_case
    r, b, _ = _row_block(p, ref)
    sf = ref["sfd_row"].copy()
    sf[orc.sf_offset(r, b, 0, p.m_pad, p.n_out // 32)] += 2
    outs = _outs(ref)
    outs["sfd_row"] = torch.from_numpy(sf)
    with pytest.raises(AssertionError, match="> 1 step"):
        compare(p, outs, ref)


def test_rows_of_another_group_fail(e4m3_case):
    p, ref = e4m3_case
    d = ref["d"].reshape(p.m_pad, -1).copy()
    d[[5, 130]] = d[[130, 5]]          # group 0 and group 2
    outs = _outs(ref)
    outs["d"] = torch.from_numpy(d.reshape(-1))
    with pytest.raises(AssertionError):
        compare(p, outs, ref)


def test_a_column_code_two_steps_off_fails(e4m3_case):
    p, ref = e4m3_case
    idx = _valid_codes(p, ref, "d_col")[:1]
    outs = _outs(ref)
    outs["d_col"] = torch.from_numpy(_bump(ref["d_col"].reshape(p.m_pad, -1), idx, 2).reshape(-1))
    with pytest.raises(AssertionError, match="D_col"):
        compare(p, outs, ref)


def test_column_scale_two_steps_off_fails(e4m3_case):
    p, ref = e4m3_case
    sf = ref["sfd_col"].copy()
    o = orc.sf_offset(7, 1, 0, p.n_out, -(-p.m_pad // 32))
    assert sf[o] > 0
    sf[o] += 2
    outs = _outs(ref)
    outs["sfd_col"] = torch.from_numpy(sf)
    with pytest.raises(AssertionError, match="D_col/SFD_col scales"):
        compare(p, outs, ref)


def test_e2m1_swapped_nibbles_fail():
    p = _problem(out_fmt="e2m1", in_fmt="nvfp4")
    ref = oracle_run(p)
    d = ref["d"].reshape(p.m_pad, -1).copy()
    lo, hi = d & 0xF, d >> 4
    far = np.abs(code_rank(lo, "e2m1") - code_rank(hi, "e2m1")) >= 2
    far[int(p.padded_offsets[-1]):] = False
    r, j = np.argwhere(far)[0]
    d[r, j] = np.uint8((int(lo[r, j]) << 4) | int(hi[r, j]))
    compare(p, _outs(ref), ref)
    outs = _outs(ref)
    outs["d"] = torch.from_numpy(d.reshape(-1))
    with pytest.raises(AssertionError, match="steps off"):
        compare(p, outs, ref)


def _bf16_bytes(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).to(torch.bfloat16).contiguous().view(torch.uint8).reshape(-1)


@pytest.mark.parametrize("rel,ok", [(0.0, True), (2.0 ** -9, True), (2.0 ** -6, False)])
def test_bf16_tolerance(rel, ok):
    p = small_problem(counts=(100, 0, 90), k=64, n=128, pad_to=32, epi="gate", out_fmt="bf16", seed=6)
    ref = oracle_run(p)
    d = np.zeros((p.m_pad, p.n_out))
    d[: ref["d_ref"].shape[0]] = ref["d_ref"] * (1.0 + rel)
    outs = {"d": _bf16_bytes(d)}
    if ok:
        compare(p, outs, ref)
    else:
        with pytest.raises(AssertionError, match="out of tolerance"):
            compare(p, outs, ref)


def test_bf16_nan_fails():
    p = small_problem(counts=(100, 0, 90), k=64, n=128, pad_to=32, epi="gate", out_fmt="bf16", seed=6)
    ref = oracle_run(p)
    d = np.zeros((p.m_pad, p.n_out))
    d[: ref["d_ref"].shape[0]] = ref["d_ref"]
    d[10, 17] = np.nan
    with pytest.raises(AssertionError, match="out of tolerance"):
        compare(p, {"d": _bf16_bytes(d)}, ref)


def test_sampled_blocks(e4m3_case):
    """The full-size tests compare a GPU run with the oracle on a list of 32-row
    blocks: the full outputs pass against the oracle's sampled run, and a
    difference inside a sampled block fails (one outside it is not looked at)."""
    p, full = e4m3_case
    blocks = np.array([0, 4, 6], dtype=np.int64)
    ref = oracle_run(p, blocks=blocks)
    compare(p, _outs(full), ref, blocks=blocks)
    for row, caught in [(4 * 32 + 3, True), (2 * 32 + 3, False)]:
        j = int(np.argwhere((full["d"].reshape(p.m_pad, -1)[row] & 0x7F) >= 0x10)[0, 0])
        outs = _outs(full)
        outs["d"] = torch.from_numpy(_bump(full["d"].reshape(p.m_pad, -1), [(row, j)], 2).reshape(-1))
        if caught:
            with pytest.raises(AssertionError, match="steps off"):
                compare(p, outs, ref, blocks=blocks)
        else:
            compare(p, outs, ref, blocks=blocks)
