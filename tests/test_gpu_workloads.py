"""Parity at full size: the four large forward workloads, the decode-like
skinny one (64 experts of a few rows each, every group one padded tile) and the
FC1 backward
(dSwiGLU, MXFP8 and the BF16 backend), generated on the GPU with their real shapes and run in every tile
shape (the library's default is the one bench.py times; two shapes for the
backward), compared element by element with the CPU oracle on
sampled 32-row blocks -- each group's first and last block, the first and last
block of the problem and random blocks -- with the same tolerances as the
small parity tests.  For BF16 outputs the per-group amax is checked over whole
groups against the GPU's own D (|amax - max|D_bf16|| <= 2^-8 amax, as D_bf16 is
D rounded to 8 significant bits), and, for the two smallest non-empty groups
of the FC2 workload, against the oracle run over every row of those groups."""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import IN_CODE, OUT_CODE, EPI_CODE, np_
from gpu_harness import TILES, tile_id, compare, decode_float_out, make_plan, run_gpu
from block_scaled_grouped_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _sample_blocks(p, n_random=12, seed=0):
    """First and last block of the problem; for the first three and last three
    non-empty groups their first block, last block and the block holding their
    last real row; a few random blocks."""
    off = np_(p.padded_offsets)
    starts = np.concatenate([[0], off[:-1]])
    nonempty = [g for g in range(p.num_groups) if off[g] > starts[g]]
    blocks = {0, p.m_pad // 32 - 1}
    for g in sorted(set(nonempty[:3] + nonempty[-3:])):
        blocks.add(int(starts[g]) // 32)
        blocks.add(int(off[g]) // 32 - 1)
        if p.counts[g] > 0:
            blocks.add(int(starts[g] + p.counts[g] - 1) // 32)
    rng = np.random.default_rng(seed)
    blocks |= set(int(b) for b in rng.integers(0, p.m_pad // 32, n_random))
    return np.array(sorted(blocks), dtype=np.int64)


def _oracle(p, blocks):
    ins = dict(a=np_(p.a), b=np_(p.b), sfa=orc.pack_sf(np_(p.sfa_rows)), sfb=orc.pack_sf(np_(p.sfb_rows)),
               padded_offsets=np_(p.padded_offsets), alpha=np_(p.alpha), prob=np_(p.prob))
    if p.epi == "dswiglu":
        ins.update(saved_c=np_(p.saved_c.double()), beta=np_(p.beta))
    if p.in_fmt == "bf16":
        ins.update(sfa=np.zeros(0, np.uint8), sfb=np.zeros(0, np.uint8))
    return orc.run(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_fmt=IN_CODE[p.in_fmt],
                   out_fmt=OUT_CODE[p.out_fmt], epi=EPI_CODE[p.epi], norm_const=p.norm_const,
                   tanh_clamp_s=p.tanh_clamp_s, want_col=p.want_col, blocks=blocks, **ins)


@pytest.fixture(scope="module", params=["fc1_swiglu", "fc2_gate", "fine_nvfp4", "skewed", "skinny"])
def workload(request):
    p = W.workload(request.param, device="cuda")
    blocks = _sample_blocks(p)
    ref = _oracle(p, blocks)
    yield p, blocks, ref
    del p
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tile", [(0, 0)] + TILES, ids=tile_id)
def test_full_size_parity_on_sampled_blocks(workload, tile):
    p, blocks, ref = workload
    outs, _, _ = run_gpu(p, tile=tile)
    compare(p, outs, ref, blocks=blocks)
    if p.out_fmt in ("bf16", "f16"):
        d = decode_float_out(outs["d"].cpu().numpy(), p.out_fmt, p.m_pad, p.n_out)
        amax = outs["amax"].cpu().numpy()
        off = np_(p.padded_offsets)
        starts = np.concatenate([[0], off[:-1]])
        for g in range(p.num_groups):
            if off[g] == starts[g]:
                assert amax[g] == 0.0
                continue
            m = np.abs(d[starts[g]:off[g]]).max()
            assert abs(amax[g] - m) <= 2.0 ** -8 * amax[g] + 1e-30, (g, amax[g], m)
        # the oracle's amax over the sampled rows bounds the full amax from below
        sampled = ref["amax"]
        assert np.all(amax >= sampled * (1 - 2.0 ** -20))


def test_full_size_group_amax_against_oracle():
    """Per-group amax of the FC2 gated workload (BF16 D, K=14336, N=4096) for
    its two smallest non-empty groups, every 32-row block of them computed by
    the oracle: within 2^-10 relative, as in the small parity tests ("Grouped
    GEMM + Quant (SM100)", Outputs: amax per group for bfloat16 D)."""
    p = W.workload("fc2_gate", device="cuda")
    off = np_(p.padded_offsets)
    starts = np.concatenate([[0], off[:-1]])
    nonempty = [g for g in range(p.num_groups) if p.counts[g] > 0]
    groups = sorted(nonempty, key=lambda g: (p.counts[g], g))[:2]
    blocks = np.concatenate([np.arange(starts[g] // 32, off[g] // 32) for g in groups]).astype(np.int64)
    ref = _oracle(p, blocks)
    outs, _, _ = run_gpu(p)
    amax = outs["amax"].cpu().numpy()
    for g in groups:
        assert ref["amax"][g] > 0.0
        np.testing.assert_allclose(amax[g], ref["amax"][g], rtol=2.0 ** -10, atol=0, err_msg=f"group {g}")
    del p, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["fc1_dswiglu", "fc1_dswiglu_bf16"])
@pytest.mark.parametrize("tile", [(0, 0), (256, 256, 2, 1)], ids=tile_id)
def test_full_size_backward_on_sampled_blocks(tile, name):
    """The FC1 + SwiGLU backward at full size (T=4096 top-2 of 8, K=4096,
    N=14336, outputs 28672 wide; MXFP8 with E4M3 row and column outputs, or
    the BF16 backend with a bfloat16 D_row): D (D_col and the scale factors) on
    sampled blocks, and dprob on every row of those blocks."""
    import block_scaled_grouped_gb300 as bsgg
    from gpu_harness import alloc_outputs, check_float_d
    p = W.workload(name, device="cuda")
    blocks = _sample_blocks(p)
    ref = _oracle(p, blocks)
    plan = bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col, tile=tuple(tile[:2]),
                     cluster=tuple(tile[2:4]) or (0, 0))
    outs = alloc_outputs(plan)
    dprob = torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=p.a, sfa=bsgg.pack_sf(p.sfa_rows), b=p.b, sfb=bsgg.pack_sf(p.sfb_rows),
             padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob, norm_const=norm,
             saved_c=p.saved_c, beta=p.beta, dprob=dprob, **outs)
    assert plan.device_status() == 0
    compare(p, outs, ref, blocks=blocks)
    rows = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    check_float_d(dprob.cpu().double().numpy()[rows], ref["dprob_ref"], what="dprob")
    del p, outs
    torch.cuda.empty_cache()
