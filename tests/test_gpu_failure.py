"""The failure path on the GPU, without a fault: with the plan's forced-timeout
hook on, the kernel's MMA thread waits on a barrier that nothing completes; every
wait is bounded (50 ms in this mode), every role gives up and returns, and the
status word reads BSGG_ERR_DEVICE_TIMEOUT.  The same plan, hook off, then runs
normally and matches the oracle: the context stays usable.  Every tile shape."""
import pytest

from helpers import oracle_run, small_problem
from gpu_harness import TILES, alloc_outputs, compare, make_plan, run_gpu, tile_id, to_device
import block_scaled_grouped_gb300 as bsgg

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("in_fmt", ["mxfp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_forced_timeout_is_reported_and_the_next_launch_is_correct(tile, in_fmt):
    p = to_device(small_problem(counts=(300, 0, 129, 500), k=512, n=256, pad_to=128, in_fmt=in_fmt,
                                epi="srelu", out_fmt="e4m3" if in_fmt != "nvfp4" else "bf16",
                                want_col=in_fmt != "nvfp4", seed=50))
    plan = make_plan(p, tile=tile)
    sfa, sfb = bsgg.pack_sf(p.sfa_rows), bsgg.pack_sf(p.sfb_rows)
    import torch
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    args = dict(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha,
                prob=p.prob, norm_const=norm)
    plan.debug_force_timeout(True)
    for _ in range(2):
        plan.run(**args, **alloc_outputs(plan))
        assert plan.device_status() == 4          # BSGG_ERR_DEVICE_TIMEOUT
    plan.debug_force_timeout(False)
    outs, _, _ = run_gpu(p, plan=plan, inputs=(sfa, sfb))
    compare(p, outs, oracle_run(p))


@pytest.mark.parametrize("in_fmt,tile", [("mxfp4", (256, 256, 2, 1)), ("fp4_ue8m0_16", (128, 128, 1, 1)),
                                         ("bf16", (128, 128, 1, 1)), ("bf16", (256, 256, 2, 1))],
                         ids=lambda x: x if isinstance(x, str) else tile_id(x))
def test_forced_timeout_other_input_classes(in_fmt, tile):
    """The same for UE8M0-scaled FP4 (scale stores) and bfloat16 operands (no
    scales: the copier idle, the MMA thread on the operands' barrier); bfloat16
    runs the dSwiGLU backward, its one epilogue family."""
    import torch
    bwd = in_fmt == "bf16"
    p = to_device(small_problem(counts=(300, 0, 129, 500), k=512, n=256, pad_to=128, in_fmt=in_fmt,
                                epi="dswiglu" if bwd else "srelu", out_fmt="bf16", seed=51))
    plan = make_plan(p, tile=tile)
    sfa, sfb = bsgg.pack_sf(p.sfa_rows), bsgg.pack_sf(p.sfb_rows)
    args = dict(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob)
    if bwd:
        args.update(saved_c=p.saved_c, beta=p.beta)
    plan.debug_force_timeout(True)
    for _ in range(2):
        extra = {"dprob": torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")} if bwd else {}
        plan.run(**args, **extra, **alloc_outputs(plan))
        assert plan.device_status() == 4          # BSGG_ERR_DEVICE_TIMEOUT
    plan.debug_force_timeout(False)
    outs = alloc_outputs(plan)
    dprob = torch.zeros(p.m_pad, dtype=torch.float32, device="cuda")
    plan.run(**args, **({"dprob": dprob} if bwd else {}), **outs)
    assert plan.device_status() == 0
    compare(p, outs, oracle_run(p))
