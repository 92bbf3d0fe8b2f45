"""bsgg_run_noalloc, the entry point for callers that cannot allocate device
memory when they call in (a framework pool that already holds the memory, a
serving loop that must not let cudaMalloc/cudaFree synchronize the device, a
plug-in whose host application owns memory).  It must give the same outputs as
the regular bsgg_run, within the parity tolerances, on two calls in a row that
share its static scratch.  This file sorts last so that a run stopping at the
first failure has run every other test already."""
import numpy as np
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from helpers import small_problem
from gpu_harness import (alloc_outputs, check_codes, check_float_d, check_sf_codes, decode_float_out,
                         make_plan, run_gpu, to_device)

pytestmark = pytest.mark.gpu

CASES = {
    "swiglu_e4m3_col": dict(counts=(200, 0, 60), k=256, n=256, epi="swiglu", out_fmt="e4m3",
                            want_col=True, seed=41),
    "gate_bf16_amax": dict(counts=(130, 256), k=384, n=256, epi="gate", out_fmt="bf16", seed=42),
    "nvfp4_srelu_e2m1": dict(counts=(128, 70), k=256, n=128, in_fmt="nvfp4", epi="srelu",
                             out_fmt="e2m1", tanh_clamp_s=8.0, seed=43),
}


def _noalloc(p, outs, sfa, sfb):
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    return bsgg.run_noalloc(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                            out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col,
                            tanh_clamp_s=p.tanh_clamp_s, wait_status=True, a=p.a, sfa=sfa, b=p.b,
                            sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob,
                            norm_const=norm, **outs)


def _same_within_tolerance(p, got, ref):
    if p.out_fmt in ("bf16", "f16", "f32"):
        d = decode_float_out(got["d"].cpu().numpy(), p.out_fmt, p.m_pad, p.n_out)
        r = decode_float_out(ref["d"].cpu().numpy(), p.out_fmt, p.m_pad, p.n_out)
        check_float_d(d, r)
        np.testing.assert_allclose(got["amax"].cpu().numpy(), ref["amax"].cpu().numpy(), rtol=2.0 ** -10)
        return
    fmt = p.out_fmt
    for name in ("d", "d_col"):
        if name in ref:
            g, r = got[name].cpu().numpy(), ref[name].cpu().numpy()
            if fmt == "e2m1":
                g = np.stack([g & 0xF, g >> 4], -1).reshape(-1)
                r = np.stack([r & 0xF, r >> 4], -1).reshape(-1)
            check_codes(g, r, fmt, name)
    for name in ("sfd_row", "sfd_col"):
        if name in ref:
            check_sf_codes(got[name].cpu().numpy(), ref[name].cpu().numpy(), name)


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_bsgg_run_on_two_calls_in_a_row(case):
    p = to_device(small_problem(pad_to=128, **CASES[case]))
    ref, sfa, sfb = run_gpu(p)                     # the regular entry point
    plan = make_plan(p)
    for _ in range(2):
        outs = alloc_outputs(plan)
        assert _noalloc(p, outs, sfa, sfb) == 0
        _same_within_tolerance(p, outs, ref)


def test_noalloc_reports_bad_offsets_and_then_recovers():
    p = to_device(small_problem(counts=(128, 128), k=128, n=128, pad_to=128, seed=44))
    ref, sfa, sfb = run_gpu(p)
    good = p.padded_offsets
    p.padded_offsets = torch.tensor([100, 256], dtype=torch.int32, device="cuda")
    outs = alloc_outputs(make_plan(p))
    assert _noalloc(p, outs, sfa, sfb) == 5        # BSGG_ERR_BAD_OFFSETS
    p.padded_offsets = good
    outs = alloc_outputs(make_plan(p))
    assert _noalloc(p, outs, sfa, sfb) == 0        # the status word was cleared
    _same_within_tolerance(p, outs, ref)
