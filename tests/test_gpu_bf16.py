"""Parity of the BF16 backend of the dGLU backward ("Grouped GEMM + dGLU
(SM100)", Backend dispatch and BF16 contract) through the C ABI against the
oracle: bfloat16 A and B without scale factors on tcgen05 kind::f16 MMAs,
ref = alpha_g^2 A B^T, X = beta_g C for dSwiGLU and dGeGLU (the source GeGLU
constants), 16/32-bit D_row, dprob and dbias accumulated into zeroed buffers;
dense and discrete (per-expert pointer) weights, every tile shape with a
bfloat16 instance, ragged groups and a K tail inside a 64-element stage.

Tolerances as everywhere: D, dprob and dbias within 2^-7 |ref| + 1e-3 rms(ref).
"""
import numpy as np
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from gpu_harness import alloc_outputs, check_float_d, compare, tile_id, to_device
from helpers import oracle_run, small_problem

pytestmark = pytest.mark.gpu

# the library's default (256 x 256 CTA pairs for the bfloat16 backward: two
# accumulators read 32 columns at a time), 128 x 128, 128 x 256 (two accumulators)
BF16_TILES = [(0, 0), (128, 128, 1, 1), (128, 256, 1, 1)]


def _run(p, tile=(0, 0), gate_first=False, saved_fmt="bf16", discrete=False, with_dbias=True):
    pd = to_device(p)
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format="bf16",
                     out_format=p.out_fmt, epilogue=p.epi, gate_first=gate_first, tile=tuple(tile[:2]),
                     cluster=tuple(tile[2:4]) or (0, 0), saved_c_format=saved_fmt, discrete_b=discrete)
    outs = alloc_outputs(plan)
    dprob = torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")
    dbias = torch.zeros(p.num_groups, 2 * p.n, dtype=torch.float32, device="cuda") if with_dbias else None
    w = {}
    keep = []
    if discrete:
        slices = [pd.b[g].clone() for g in range(p.num_groups)]
        keep.append(slices)
        w["b_ptrs"] = torch.tensor([0 if p.counts[g] == 0 else slices[g].data_ptr()
                                    for g in range(p.num_groups)], dtype=torch.int64, device="cuda")
    else:
        w["b"] = pd.b
    plan.run(a=pd.a, padded_offsets=pd.padded_offsets, alpha=pd.alpha, prob=pd.prob, saved_c=pd.saved_c,
             beta=pd.beta, dprob=dprob, dbias=dbias, **w, **outs)
    assert plan.device_status() == 0
    ref = oracle_run(p, gate_first=int(gate_first))
    compare(p, outs, ref)
    np.testing.assert_allclose(outs["amax"].cpu().numpy(), ref["amax"], rtol=2.0 ** -10, atol=0)
    check_float_d(dprob.cpu().double().numpy(), ref["dprob_ref"], what="dprob")
    if with_dbias:
        check_float_d(dbias.cpu().double().numpy(), ref["dbias"], what="dbias")
    return outs, ref


@pytest.mark.parametrize("gate_first", [False, True])
@pytest.mark.parametrize("tile", BF16_TILES, ids=tile_id)
def test_bf16_dswiglu(tile, gate_first):
    # K = 200: three full 64-element stages and an 8-element tail
    p = small_problem(counts=(130, 0, 256, 40), k=200, n=256, pad_to=128, in_fmt="bf16", epi="dswiglu",
                      out_fmt="bf16", seed=110)
    _run(p, tile, gate_first)


@pytest.mark.parametrize("tile", BF16_TILES, ids=tile_id)
def test_bf16_dgeglu_reads_beta_and_clamps(tile):
    # saved C ~ N(0, 8): values beyond the +-7 clamps; beta ~ U(0.5, 2) scales C first
    p = small_problem(counts=(150, 0, 300), k=256, n=128, pad_to=128, in_fmt="bf16", epi="dgeglu",
                      out_fmt="f32", seed=111)
    p.saved_c = (p.saved_c.float() * 4.0).to(torch.bfloat16)
    _run(p, tile)


@pytest.mark.parametrize("saved_fmt", ["f16", "f32"])
def test_bf16_saved_c_formats_and_f16_out(saved_fmt):
    p = small_problem(counts=(128, 150), k=128, n=128, pad_to=128, in_fmt="bf16", epi="dswiglu",
                      out_fmt="f16", seed=112)
    p.saved_c = p.saved_c.to(torch.float16 if saved_fmt == "f16" else torch.float32)
    _run(p, saved_fmt=saved_fmt)


@pytest.mark.parametrize("tile", [(0, 0), (128, 128, 1, 1)], ids=tile_id)
def test_bf16_discrete_equals_dense(tile):
    p = small_problem(counts=(0, 200, 129, 0), k=192, n=128, pad_to=128, in_fmt="bf16", epi="dgeglu",
                      out_fmt="bf16", seed=113)
    dense, _ = _run(p, tile, with_dbias=False)
    disc, _ = _run(p, tile, discrete=True, with_dbias=False)
    assert torch.equal(dense["d"], disc["d"])
