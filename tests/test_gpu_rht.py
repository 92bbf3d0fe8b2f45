"""Parity of the rowwise Hadamard output ("Grouped GEMM + GLU + Hadamard +
Quant (SM100)", Equations: H16 / 4 applied to every 16-column block of
bf16-rounded D) through the C ABI against the oracle, in every tile shape:
bf16 RHT within the D tolerance plus the effect of bf16 rounding decisions
taken on differently rounded D (see _check_bf16_rht), and exactly H/4 of the
kernel's own bf16 D where D is bf16; NVFP4 RHT codes and E4M3 SFRHT scales
>= 99.9% bit-equal (the rest one step); D still matches.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import block_scaled_grouped_gb300 as bsgg
import oracle as orc
from gpu_harness import (TILES, _check_quant_plane, alloc_outputs, check_float_d, compare, decode_float_out,
                         tile_id, to_device, unpack_e2m1)
from helpers import oracle_run, small_problem

pytestmark = pytest.mark.gpu


def _check_bf16_rht(got, ref, d_ref):
    """The D tolerance, plus what bf16 rounding decisions taken on fp32 (kernel)
    and fp64 (oracle) values of D allow: an input of a block that lands next to
    a bf16 tie may round to the neighbouring value on one side, which moves each
    of the block's 16 outputs by a quarter of that input's bf16 step (at most
    2^-7 of the block's largest input); up to two such inputs per block."""
    rows, nd = ref.shape
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    blk = np.repeat(np.abs(d_ref).reshape(rows, -1, 16).max(-1), 16, axis=1)
    tol = 2.0 ** -7 * np.abs(ref) + 1e-3 * rms + 2 * 2.0 ** -7 * blk / 4
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), f"RHT: {int(bad.sum())} of {bad.size} out of tolerance"


def _check_colwise(p, outs, ref, rht_norm):
    """Per expert: the (n_out, expert_m) code matrix and its per-16-token scales
    of the GPU against the oracle's, by the quantized-output rule."""
    nd = p.n_out
    off = np.asarray(p.padded_offsets.cpu())
    gq_all = outs["rht"].cpu().numpy()
    gs_all = outs["sfrht"].cpu().numpy()
    nib = lambda b: np.stack([b & 0xF, b >> 4], -1).reshape(-1)
    g_codes, r_codes = nib(gq_all), nib(ref["rht_q"])
    start = 0
    for g in range(p.num_groups):
        em = int(off[g]) - start
        if em == 0:
            continue
        e0 = nd * start
        gq = g_codes[e0:e0 + nd * em].reshape(nd, em)
        rq = r_codes[e0:e0 + nd * em].reshape(nd, em)
        offs = np.array([[nd * start // 16 + orc.sf_offset(n, b, 0, nd, em // 16) for b in range(em // 16)]
                         for n in range(nd)])
        y = ref["rht_ref"][start:start + em].T                 # (n_out, expert_m)
        _check_quant_plane(gq, rq, gs_all[offs], ref["sfrht"][offs], y, "e2m1", "nvfp4", rht_norm, 16, 1,
                           f"colwise RHT expert {g}")
        start = int(off[g])


def _run(p, tile, rht_format, rht_norm=1.0, **desc):
    pd = to_device(p)
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col, tanh_clamp_s=p.tanh_clamp_s,
                     tile=tuple(tile[:2]), cluster=tuple(tile[2:4]) or (0, 0), rht_format=rht_format, **desc)
    outs = alloc_outputs(plan)
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    rnorm = torch.tensor([rht_norm], dtype=torch.float32, device="cuda")
    plan.run(a=pd.a, sfa=bsgg.pack_sf(pd.sfa_rows), b=pd.b, sfb=bsgg.pack_sf(pd.sfb_rows),
             padded_offsets=pd.padded_offsets, alpha=pd.alpha, prob=pd.prob, norm_const=norm,
             rht_norm_const=rnorm, **outs)
    assert plan.device_status() == 0
    over = {}
    if "glu_limit" in desc:
        over["glu_limit"] = desc["glu_limit"]
    colwise = desc.get("rht_colwise", False)
    ref = oracle_run(p, rht="col_e2m1" if colwise else rht_format, rht_norm=rht_norm, **over)
    compare(p, outs, ref)
    nd = p.n_out
    if colwise:
        _check_colwise(p, outs, ref, rht_norm)
    elif rht_format == "bf16":
        got = decode_float_out(outs["rht"].cpu().numpy(), "bf16", p.m_pad, nd)
        _check_bf16_rht(got, ref["rht_ref"], ref["d_ref"])
        if p.out_fmt == "bf16":
            # the kernel's bf16 D is exactly the transform's input: the RHT must
            # be H/4 of it up to the fp32 sums and the bf16 output rounding
            x = decode_float_out(outs["d"].cpu().numpy(), "bf16", p.m_pad, nd)
            H = scipy.linalg.hadamard(16) / 4.0
            want = (x.reshape(p.m_pad, -1, 16) @ H.T).reshape(p.m_pad, nd)
            blk = np.abs(x.reshape(p.m_pad, -1, 16)).max(-1, keepdims=True)
            err = np.abs(got - want).reshape(p.m_pad, -1, 16)
            assert np.all(err <= 2.0 ** -8 * np.abs(want.reshape(err.shape)) + 1e-6 * blk)
    else:
        g = unpack_e2m1(outs["rht"].cpu().numpy(), p.m_pad, nd)
        r = unpack_e2m1(ref["rht_q"], p.m_pad, nd)
        kb = nd // 16
        offs = np.array([[orc.sf_offset(m, j, 0, p.m_pad, kb) for j in range(kb)] for m in range(p.m_pad)])
        _check_quant_plane(g, r, outs["sfrht"].cpu().numpy()[offs], ref["sfrht"][offs], ref["rht_ref"], "e2m1",
                           "nvfp4", rht_norm, 16, 1, "RHT/SFRHT")
    return outs, ref


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_swiglu_e2m1_d_and_e2m1_rht(tile):
    p = small_problem(counts=(150, 0, 300), k=512, n=512, pad_to=128, in_fmt="nvfp4", epi="swiglu",
                      out_fmt="e2m1", seed=80)
    _run(p, tile, "e2m1", rht_norm=0.5)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_mxfp8_gate_bf16_rht(tile):
    p = small_problem(counts=(200, 77), k=256, n=256, pad_to=128, epi="gate", out_fmt="bf16", seed=81)
    _run(p, tile, "bf16")


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_geglu_srelu_with_rht_bias_and_c(tile):
    # the Hadamard output together with the other extended outputs
    p = small_problem(counts=(128, 60), k=256, n=256, pad_to=128, in_fmt="nvfp4", epi="geglu",
                      out_fmt="bf16", seed=82)
    _run(p, tile, "e2m1", rht_norm=2.0, glu_limit=9.0)
    p = small_problem(counts=(128, 60), k=256, n=128, pad_to=128, epi="srelu", out_fmt="e4m3",
                      want_col=True, tanh_clamp_s=8.0, seed=83)
    _run(p, tile, "bf16")


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_colwise_rht_nvfp4(tile):
    # experts of 256, 0, 384 and 128 padded rows; N_out = 256
    p = small_problem(counts=(150, 0, 300, 128), k=512, n=512, pad_to=128, in_fmt="nvfp4", epi="swiglu",
                      out_fmt="e2m1", seed=84)
    _run(p, tile, "e2m1", rht_norm=0.5, rht_colwise=True)
    p = small_problem(counts=(200, 77), k=256, n=256, pad_to=128, epi="srelu", out_fmt="e4m3",
                      want_col=True, tanh_clamp_s=8.0, seed=85)
    _run(p, tile, "e2m1", rht_norm=2.0, rht_colwise=True)
