"""Parity of the dSwiGLU, dGeGLU and dSiTU-GLU backward ("Grouped GEMM + dGLU
(SM100)", Block-scaled contract) through the C ABI against the oracle, in every
tile shape: the
2N-wide interleaved input/gate gradients (16/32-bit with the two amax halves,
or FP8/FP4 with row and column scale factors), and dprob, which the kernel
accumulates into the caller's zeroed buffer.

Tolerances: D as everywhere (2^-7 |ref| + 1e-3 rms(ref) for 16/32-bit, >= 99.9%
bit-equal codes otherwise); dprob within 2^-7 |ref| + 1e-3 rms(ref) (an fp32
sum over N products, in a different order than the oracle's fp64 sum).
"""
import numpy as np
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from gpu_harness import TILES, alloc_outputs, check_float_d, compare, tile_id, to_device
from helpers import oracle_run, small_problem

pytestmark = pytest.mark.gpu


def _run(p, tile=(0, 0), gate_first=False, saved_fmt="bf16", dprob=None, dgeglu_params=None, situ_betas=None):
    pd = to_device(p)
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col, gate_first=gate_first,
                     tile=tuple(tile[:2]), cluster=tuple(tile[2:4]) or (0, 0), saved_c_format=saved_fmt,
                     dgeglu_params=dgeglu_params, situ_betas=situ_betas)
    outs = alloc_outputs(plan)
    if dprob is None:
        dprob = torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=pd.a, sfa=bsgg.pack_sf(pd.sfa_rows), b=pd.b, sfb=bsgg.pack_sf(pd.sfb_rows),
             padded_offsets=pd.padded_offsets, alpha=pd.alpha, prob=pd.prob, norm_const=norm,
             saved_c=pd.saved_c, beta=pd.beta if p.epi == "dswiglu" else None, dprob=dprob, **outs)
    assert plan.device_status() == 0
    return plan, outs, dprob


def _check(p, outs, dprob, gate_first=False, dgeglu_params=None, situ_betas=None):
    over = {}
    if dgeglu_params is not None:
        over = dict(zip(("geglu_alpha", "glu_clamp_min", "glu_clamp_max", "linear_offset"), dgeglu_params))
    if situ_betas is not None:
        over.update(situ_beta1=situ_betas[0], situ_beta2=situ_betas[1])
    ref = oracle_run(p, gate_first=int(gate_first), **over)
    compare(p, outs, ref)
    if "amax" in outs:
        np.testing.assert_allclose(outs["amax"].cpu().numpy(), ref["amax"], rtol=2.0 ** -10, atol=0)
    check_float_d(dprob.cpu().double().numpy(), ref["dprob_ref"], what="dprob")
    return ref


@pytest.mark.parametrize("gate_first", [False, True])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dswiglu_bf16_ragged(tile, gate_first):
    p = small_problem(counts=(130, 0, 256, 40), k=256, n=256, pad_to=128, epi="dswiglu", out_fmt="bf16",
                      seed=70)
    plan, outs, dprob = _run(p, tile, gate_first)
    _check(p, outs, dprob, gate_first)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dswiglu_e4m3_row_and_col_n_tail(tile):
    # N = 96: the last n-tile of 128 or 256 columns is mostly past N
    p = small_problem(counts=(200, 77), k=384, n=96, pad_to=128, epi="dswiglu", out_fmt="e4m3",
                      want_col=True, seed=71)
    plan, outs, dprob = _run(p, tile)
    _check(p, outs, dprob)


@pytest.mark.parametrize("saved_fmt", ["f16", "f32"])
def test_dswiglu_saved_c_formats(saved_fmt):
    p = small_problem(counts=(128, 150), k=256, n=128, pad_to=128, epi="dswiglu", out_fmt="f32", seed=72)
    p.saved_c = p.saved_c.to(torch.float16 if saved_fmt == "f16" else torch.float32)
    plan, outs, dprob = _run(p, saved_fmt=saved_fmt)
    _check(p, outs, dprob)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dswiglu_nvfp4_e2m1_and_bf16(tile):
    p = small_problem(counts=(150, 0, 300), k=512, n=256, pad_to=128, in_fmt="nvfp4", epi="dswiglu",
                      out_fmt="e2m1", want_col=True, seed=73)
    plan, outs, dprob = _run(p, tile)
    _check(p, outs, dprob)
    p = small_problem(counts=(128, 60), k=256, n=128, pad_to=128, in_fmt="nvfp4", epi="dswiglu",
                      out_fmt="bf16", seed=74)
    plan, outs, dprob = _run(p, tile)
    _check(p, outs, dprob)


@pytest.mark.parametrize("in_fmt", ["fp4_ue8m0_16", "mxfp4"])
@pytest.mark.parametrize("tile", [(0, 0), (256, 256, 2, 1)], ids=tile_id)
def test_dswiglu_fp4_with_ue8m0_scales(tile, in_fmt):
    p = small_problem(counts=(150, 0, 300), k=544, n=256, pad_to=128, in_fmt=in_fmt, epi="dswiglu",
                      out_fmt="e2m1", want_col=True, seed=75)
    plan, outs, dprob = _run(p, tile)
    _check(p, outs, dprob)


def test_dprob_accumulates_and_zero_prob_rows_still_get_it():
    p = small_problem(counts=(128, 100), k=256, n=128, pad_to=128, epi="dswiglu", out_fmt="bf16", seed=75)
    p.prob[:64] = 0.0                        # routing weight 0: D rows 0, dprob not
    plan, outs, dprob = _run(p)
    ref = _check(p, outs, dprob)
    once = dprob.clone()
    assert torch.all(once[:64] != 0)
    # a second call adds to the caller's buffer
    plan2, outs2, dprob2 = _run(p, dprob=dprob)
    check_float_d(dprob2.cpu().double().numpy(), 2 * ref["dprob_ref"], what="dprob (twice)")


def test_backward_requires_its_inputs():
    p = to_device(small_problem(counts=(128,), k=128, n=128, pad_to=128, epi="dswiglu", seed=76))
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=1, in_format=p.in_fmt, out_format="bf16",
                     epilogue="dswiglu")
    outs = alloc_outputs(plan)
    base = dict(a=p.a, sfa=bsgg.pack_sf(p.sfa_rows), b=p.b, sfb=bsgg.pack_sf(p.sfb_rows),
                padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob, **outs)
    dprob = torch.zeros(p.m_pad, device="cuda")
    for missing in ("saved_c", "beta", "dprob"):
        extra = dict(saved_c=p.saved_c, beta=p.beta, dprob=dprob)
        extra.pop(missing)
        with pytest.raises(bsgg.BsggError) as e:
            plan.run(**base, **extra)
        assert e.value.code == 1


@pytest.mark.parametrize("gate_first", [False, True])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dgeglu_bf16_with_clamped_values(tile, gate_first):
    # saved C ~ N(0, 8): many values beyond the +-7 clamp, masks and clamps hit
    p = small_problem(counts=(130, 0, 256, 40), k=256, n=256, pad_to=128, epi="dgeglu", out_fmt="bf16",
                      seed=90)
    p.saved_c = (p.saved_c.float() * 4.0).to(torch.bfloat16)
    plan, outs, dprob = _run(p, tile, gate_first)
    _check(p, outs, dprob, gate_first)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dgeglu_custom_params_e4m3(tile):
    # the clamped-SwiGLU configuration the page gives: alpha 1, offset 0, +-10
    params = (1.0, -10.0, 10.0, 0.0)
    p = small_problem(counts=(200, 77), k=384, n=96, pad_to=128, epi="dgeglu", out_fmt="e4m3",
                      want_col=True, seed=91)
    p.saved_c = (p.saved_c.float() * 5.0).to(torch.bfloat16)
    plan, outs, dprob = _run(p, tile, dgeglu_params=params)
    _check(p, outs, dprob, dgeglu_params=params)


def test_dgeglu_nvfp4_f16_saved_c():
    p = small_problem(counts=(150, 0, 300), k=512, n=128, pad_to=128, in_fmt="nvfp4", epi="dgeglu",
                      out_fmt="e2m1", want_col=True, seed=92)
    p.saved_c = (p.saved_c.float() * 4.0).to(torch.float16)
    plan, outs, dprob = _run(p, saved_fmt="f16")
    _check(p, outs, dprob)


@pytest.mark.parametrize("betas", [None, (2.0, 0.5)], ids=["unit", "b2_05"])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dsituglu_e4m3_and_bf16(tile, betas):
    p = small_problem(counts=(130, 0, 256, 40), k=256, n=128, pad_to=128, epi="dsituglu", out_fmt="e4m3",
                      want_col=True, seed=93)
    plan, outs, dprob = _run(p, tile, situ_betas=betas)
    _check(p, outs, dprob, situ_betas=betas)
    p = small_problem(counts=(200, 77), k=384, n=96, pad_to=128, epi="dsituglu", out_fmt="bf16", seed=94)
    plan, outs, dprob = _run(p, tile, situ_betas=betas)
    _check(p, outs, dprob, situ_betas=betas)


@pytest.mark.parametrize("epi", ["dswiglu", "dgeglu", "dsituglu"])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_dbias_row_sums_per_group(tile, epi):
    """dbias (L, 2N) accumulates the rows of D of each group (caller-zeroed),
    within 2^-7 |ref| + 1e-3 rms(ref) of the oracle's fp64 sums; D and dprob
    are unchanged by asking for it."""
    p = small_problem(counts=(130, 0, 256, 40), k=256, n=128, pad_to=128, epi=epi, out_fmt="e4m3",
                      want_col=True, seed=95)
    pd = to_device(p)
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=epi, want_col=True, tile=tuple(tile[:2]),
                     cluster=tuple(tile[2:4]) or (0, 0))
    outs = alloc_outputs(plan)
    dprob = torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")
    dbias = torch.zeros(p.num_groups, 2 * p.n, dtype=torch.float32, device="cuda")
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=pd.a, sfa=bsgg.pack_sf(pd.sfa_rows), b=pd.b, sfb=bsgg.pack_sf(pd.sfb_rows),
             padded_offsets=pd.padded_offsets, alpha=pd.alpha, prob=pd.prob, norm_const=norm,
             saved_c=pd.saved_c, beta=pd.beta if epi == "dswiglu" else None, dprob=dprob, dbias=dbias, **outs)
    assert plan.device_status() == 0
    ref = _check(p, outs, dprob)
    check_float_d(dbias.cpu().double().numpy(), ref["dbias"], what="dbias")
    assert torch.all(dbias[1] == 0)                  # the empty group


def test_dbias_only_with_a_backward_epilogue():
    p = to_device(small_problem(counts=(128,), k=128, n=128, pad_to=128, seed=96))
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=1, in_format=p.in_fmt, out_format="bf16",
                     epilogue="gate")
    outs = alloc_outputs(plan)
    with pytest.raises(bsgg.BsggError) as e:
        plan.run(a=p.a, sfa=bsgg.pack_sf(p.sfa_rows), b=p.b, sfb=bsgg.pack_sf(p.sfb_rows),
                 padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob,
                 dbias=torch.zeros(1, 128, device="cuda"), **outs)
    assert e.value.code == 1
