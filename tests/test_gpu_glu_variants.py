"""Parity of the forward epilogue options of "Grouped GEMM + GLU + Hadamard +
Quant (SM100)", Equations, through the C ABI against the oracle: the per-expert
bias added to C, the stored pre-activation C (bf16 / f16), GeGLU, and the GLU
clamp (glu_limit) and output scale (glu_alpha), in every tile shape.

Tolerances as for D: C and 16/32-bit D within 2^-7 |ref| + 1e-3 rms(ref);
quantized D and scale factors bit-equal on >= 99.9%, the rest one code step.
"""
import numpy as np
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from gpu_harness import TILES, alloc_outputs, check_float_d, compare, decode_float_out, tile_id, to_device
from helpers import oracle_run, small_problem

pytestmark = pytest.mark.gpu


def _bias(p, fmt, seed):
    """(L, N) bias drawn N(0, 4) and rounded to `fmt`; returns (device tensor
    in fmt, the same values as float32 for the oracle)."""
    g = np.random.default_rng(seed)
    b = torch.from_numpy(g.normal(0.0, 4.0, size=(p.num_groups, p.n)).astype(np.float32))
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[fmt]
    bq = b.to(dt)
    return bq.cuda().contiguous(), bq.float().numpy()


def _run(p, tile, *, gate_first=False, glu_limit=0.0, glu_alpha=0.0, c_format=None, bias_format=None,
         seed=0):
    pd = to_device(p)
    cluster = tuple(tile[2:4])
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col, gate_first=gate_first,
                     tanh_clamp_s=p.tanh_clamp_s, tile=tuple(tile[:2]), cluster=cluster,
                     glu_limit=glu_limit, glu_alpha=glu_alpha, c_format=c_format,
                     bias_format=bias_format)
    outs = alloc_outputs(plan)
    extra, over = {}, {}
    if bias_format is not None:
        extra["bias"], over["bias"] = _bias(p, bias_format, seed)
    sfa, sfb = bsgg.pack_sf(pd.sfa_rows), bsgg.pack_sf(pd.sfb_rows)
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=pd.a, sfa=sfa, b=pd.b, sfb=sfb, padded_offsets=pd.padded_offsets, alpha=pd.alpha,
             prob=pd.prob, norm_const=norm, **extra, **outs)
    assert plan.device_status() == 0
    ref = oracle_run(p, gate_first=int(gate_first), glu_limit=glu_limit,
                     glu_alpha=(glu_alpha if glu_alpha != 0.0 else 1.0), want_c=c_format is not None, **over)
    compare(p, outs, ref)
    if "amax" in outs:
        np.testing.assert_allclose(outs["amax"].cpu().numpy(), ref["amax"], rtol=2.0 ** -10, atol=0)
    if c_format in ("bf16", "f16", "f32"):
        c = decode_float_out(outs["c"].cpu().numpy(), c_format, p.m_pad, p.n)
        check_float_d(c, ref["c_ref"], what="C")
    elif c_format is not None:
        _check_quantized_c(outs["c"].cpu().numpy(), ref["c_ref"], c_format, p.m_pad, p.n)
    return outs, ref


def _check_quantized_c(raw, c_ref, fmt, m_pad, n):
    """FP8 / FP4 C without a scale factor: the codes equal the oracle's
    round-to-nearest-even saturating encoding of its fp64 C (rounded to fp32,
    the precision the kernel converts from) on >= 99.9 % of the elements, and
    every code decodes within one code step of C (the kernel's C is an fp32 sum
    in another order)."""
    import oracle as orc
    code_fmt = {"e4m3": 0, "e5m2": 1, "e2m1": 2}[fmt]
    if fmt == "e2m1":
        codes = np.stack([raw & 0xF, raw >> 4], axis=-1).reshape(m_pad, n)
    else:
        codes = raw.reshape(m_pad, n)
    rows = c_ref.shape[0]
    want = np.array([[orc.encode_rne_satfinite(code_fmt, float(np.float32(x))) for x in r] for r in c_ref])
    got = codes[:rows]
    match = np.mean(got == want)
    assert match >= 0.999, (fmt, match)
    dec = np.vectorize(lambda c: orc.decode(code_fmt, int(c)))
    g, w = dec(got), dec(want)
    step = {"e4m3": 2.0 ** -3, "e5m2": 2.0 ** -2, "e2m1": 0.5}[fmt]
    assert np.all(np.abs(g - w) <= step * np.maximum(np.abs(w), 1.0) + 1e-30)


@pytest.mark.parametrize("gate_first", [False, True])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_geglu_e4m3_bias_clamp_scale_and_c(tile, gate_first):
    p = small_problem(counts=(130, 256, 0, 40), k=256, n=512, pad_to=128, epi="geglu", out_fmt="e4m3",
                      want_col=True, seed=50)
    _run(p, tile, gate_first=gate_first, glu_limit=10.0, glu_alpha=0.75, c_format="bf16",
         bias_format="f32", seed=1)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_swiglu_bf16_clamp_scale_bf16_bias_f16_c(tile):
    p = small_problem(counts=(200, 0, 77), k=384, n=256, pad_to=128, epi="swiglu", out_fmt="bf16",
                      seed=51)
    _run(p, tile, glu_limit=7.0, glu_alpha=1.5, c_format="f16", bias_format="bf16", seed=2)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_geglu_bf16_without_options(tile):
    p = small_problem(counts=(128, 300), k=256, n=256, pad_to=128, epi="geglu", out_fmt="bf16", seed=52)
    _run(p, tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_gate_bf16_with_f16_bias_and_c_and_n_tail(tile):
    # N = 96: the last n-tile is mostly past N (no C stored, no bias read there)
    p = small_problem(counts=(300, 0, 129), k=256, n=96, pad_to=128, epi="gate", out_fmt="bf16", seed=53)
    _run(p, tile, c_format="bf16", bias_format="f16", seed=3)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_c_only_srelu_e4m3(tile):
    p = small_problem(counts=(256, 70), k=256, n=256, pad_to=128, epi="srelu", out_fmt="e4m3",
                      want_col=True, tanh_clamp_s=8.0, seed=54)
    _run(p, tile, c_format="bf16")


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_geglu_e2m1_bias_and_c(tile):
    p = small_problem(counts=(150, 0, 300), k=512, n=512, pad_to=128, in_fmt="nvfp4", epi="geglu",
                      out_fmt="e2m1", want_col=True, seed=55)
    _run(p, tile, glu_limit=12.0, c_format="bf16", bias_format="bf16", seed=4)


@pytest.mark.parametrize("c_format", ["f32", "e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("tile", [(128, 128, 1, 1), (256, 256, 2, 1)], ids=tile_id)
def test_mxfp8_c_in_f32_fp8_and_fp4(tile, c_format):
    # "Grouped GEMM + SwiGLU (SM100)" / "Grouped GEMM + sReLU (SM100)": with FP8
    # inputs C may be f32, e4m3, e5m2 or e2m1 (no scale factor for C)
    p = small_problem(counts=(130, 0, 256), k=256, n=256, pad_to=128, epi="swiglu", out_fmt="e4m3",
                      seed=6)
    _run(p, tile, c_format=c_format, bias_format="f32", seed=6)


def test_bias_and_c_required_when_described():
    p = to_device(small_problem(counts=(128,), k=128, n=128, pad_to=128, seed=56))
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=1, in_format=p.in_fmt, out_format="bf16",
                     epilogue="gate", c_format="bf16", bias_format="f32")
    outs = alloc_outputs(plan)
    sfa, sfb = bsgg.pack_sf(p.sfa_rows), bsgg.pack_sf(p.sfb_rows)
    base = dict(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha,
                prob=p.prob)
    c = outs.pop("c")
    bias = torch.zeros(1, p.n, device="cuda")
    with pytest.raises(bsgg.BsggError) as e:
        plan.run(**base, **outs, c=c)             # bias missing
    assert e.value.code == 1
    with pytest.raises(bsgg.BsggError) as e:
        plan.run(**base, **outs, bias=bias)       # C missing
    assert e.value.code == 1
    with pytest.raises(bsgg.BsggError) as e:      # C misaligned
        plan.run(**base, **outs, bias=bias, c=c[8:])
    assert e.value.code == 1
