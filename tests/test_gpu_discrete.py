"""Discrete weight mode ("Grouped GEMM + GLU + Hadamard + Quant (SM100)",
Discrete weight mode) through the C ABI: each expert's B and SFB are separate
allocations named by device arrays of pointers.  The outputs must equal the
dense-mode outputs of the same problem bit for bit (same arithmetic in the
same order) and match the oracle within the usual tolerances.  Pointers of
empty groups may be 0; a bad pointer of a non-empty group is reported as
BSGG_ERR_BAD_POINTERS and nothing is written.
"""
import numpy as np
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from gpu_harness import SENTINEL, TILES, alloc_outputs, compare, tile_id, to_device
from helpers import oracle_run, small_problem

pytestmark = pytest.mark.gpu


def _plan(p, tile, discrete):
    return bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col,
                     tanh_clamp_s=p.tanh_clamp_s, tile=tuple(tile[:2]),
                     cluster=tuple(tile[2:4]) or (0, 0), discrete_b=discrete)


def _expert_buffers(p, null_empty=True):
    """One allocation per expert for B_g and SFB_g; the pointer arrays (0 for
    empty groups when null_empty)."""
    counts = p.counts
    bs, sfbs, bp, sp = [], [], [], []
    for g in range(p.num_groups):
        b = p.b[g].clone()
        sfb = bsgg.pack_sf(p.sfb_rows[g:g + 1].contiguous())
        bs.append(b)
        sfbs.append(sfb)
        empty = counts[g] == 0
        bp.append(0 if (empty and null_empty) else b.data_ptr())
        sp.append(0 if (empty and null_empty) else sfb.data_ptr())
    b_ptrs = torch.tensor(bp, dtype=torch.int64, device="cuda")
    sfb_ptrs = torch.tensor(sp, dtype=torch.int64, device="cuda")
    return (bs, sfbs), b_ptrs, sfb_ptrs


def _run(plan, p, sfa, outs, **w):
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=p.a, sfa=sfa, padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob,
             norm_const=norm, **w, **outs)
    return plan.device_status()


CASES = {
    "mxfp8_swiglu_e4m3": dict(counts=(130, 0, 256, 40), k=384, n=512, epi="swiglu", out_fmt="e4m3",
                              want_col=True, seed=60),
    "mxfp8_gate_bf16": dict(counts=(0, 300, 129, 0), k=256, n=384, seed=61),
    "nvfp4_srelu_e2m1": dict(counts=(150, 0, 300), k=512, n=256, in_fmt="nvfp4", epi="srelu",
                             out_fmt="e2m1", tanh_clamp_s=8.0, seed=62),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_discrete_equals_dense_and_oracle(tile, case):
    p = to_device(small_problem(pad_to=128, **CASES[case]))
    sfa = bsgg.pack_sf(p.sfa_rows)
    dense = _plan(p, tile, False)
    o_dense = alloc_outputs(dense)
    assert _run(dense, p, sfa, o_dense, b=p.b, sfb=bsgg.pack_sf(p.sfb_rows)) == 0
    disc = _plan(p, tile, True)
    keep, b_ptrs, sfb_ptrs = _expert_buffers(p)
    for rep in range(2):                       # the maps are rewritten on every launch
        o_disc = alloc_outputs(disc)
        assert _run(disc, p, sfa, o_disc, b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs) == 0
        for name, t in o_dense.items():
            assert torch.equal(t, o_disc[name]), name
    compare(p, o_disc, oracle_run(p))


def test_discrete_weights_follow_the_pointers():
    # swapping two experts' pointers equals swapping their dense slices
    p = to_device(small_problem(counts=(200, 130), k=256, n=256, pad_to=128, seed=63))
    sfa = bsgg.pack_sf(p.sfa_rows)
    keep, b_ptrs, sfb_ptrs = _expert_buffers(p)
    disc = _plan(p, (0, 0), True)
    o_disc = alloc_outputs(disc)
    assert _run(disc, p, sfa, o_disc, b_ptrs=b_ptrs.flip(0).contiguous(),
                sfb_ptrs=sfb_ptrs.flip(0).contiguous()) == 0
    dense = _plan(p, (0, 0), False)
    o_dense = alloc_outputs(dense)
    assert _run(dense, p, sfa, o_dense, b=p.b.flip(0).contiguous(),
                sfb=bsgg.pack_sf(p.sfb_rows.flip(0).contiguous())) == 0
    for name, t in o_dense.items():
        assert torch.equal(t, o_disc[name]), name


@pytest.mark.parametrize("which", ["b_null", "sfb_misaligned"])
def test_bad_pointer_reported_and_nothing_written(which):
    p = to_device(small_problem(counts=(128, 0, 256), k=128, n=128, pad_to=128, seed=64))
    sfa = bsgg.pack_sf(p.sfa_rows)
    keep, b_ptrs, sfb_ptrs = _expert_buffers(p)
    if which == "b_null":
        b_ptrs[2] = 0
    else:
        sfb_ptrs[0] += 8
    plan = _plan(p, (0, 0), True)
    outs = alloc_outputs(plan)
    assert _run(plan, p, sfa, outs, b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs) == 6
    assert (outs["d"] == SENTINEL).all()
    # the plan stays usable: good pointers next
    keep2, b_ptrs, sfb_ptrs = _expert_buffers(p)
    assert _run(plan, p, sfa, outs, b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs) == 0
    compare(p, outs, oracle_run(p))


def test_dense_and_discrete_are_exclusive():
    p = to_device(small_problem(counts=(128,), k=128, n=128, pad_to=128, seed=65))
    sfa, sfb = bsgg.pack_sf(p.sfa_rows), bsgg.pack_sf(p.sfb_rows)
    keep, b_ptrs, sfb_ptrs = _expert_buffers(p)
    disc, dense = _plan(p, (0, 0), True), _plan(p, (0, 0), False)
    outs = alloc_outputs(dense)
    for plan, w in ((disc, dict(b=p.b, sfb=sfb, b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs)),
                    (disc, dict(b_ptrs=b_ptrs)),
                    (dense, dict(b=p.b, sfb=sfb, b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs))):
        with pytest.raises(bsgg.BsggError) as e:
            _run(plan, p, sfa, outs, **w)
        assert e.value.code == 1
    # the allocation-free entry point cannot hold per-expert descriptors
    code = bsgg.run_noalloc(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=1, in_format=p.in_fmt,
                            out_format=p.out_fmt, epilogue=p.epi, discrete_b=True, a=p.a, sfa=sfa,
                            b_ptrs=b_ptrs, sfb_ptrs=sfb_ptrs, padded_offsets=p.padded_offsets,
                            alpha=p.alpha, prob=p.prob, **outs)
    assert code == 2
