"""bsgg_run inside a captured CUDA graph: one warm-up launch, capture, two
replays; the outputs equal an eager launch's bit for bit (same kernel, same
inputs), and the amax reset inside the graph works on every replay."""
import pytest
import torch

import block_scaled_grouped_gb300 as bsgg
from helpers import small_problem
from gpu_harness import alloc_outputs, make_plan, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["gate_bf16", "swiglu_e4m3"])
def test_graph_replay_matches_eager(case):
    if case == "gate_bf16":
        p = to_device(small_problem(counts=(200, 300), k=512, n=256, pad_to=128, seed=51))
    else:
        p = to_device(small_problem(counts=(200, 300), k=512, n=256, pad_to=128, epi="swiglu",
                                    out_fmt="e4m3", want_col=True, seed=52))
    plan = make_plan(p)
    sfa, sfb = bsgg.pack_sf(p.sfa_rows), bsgg.pack_sf(p.sfb_rows)
    norm = torch.ones(1, device="cuda")
    ins = dict(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha,
               prob=p.prob, norm_const=norm)
    eager = alloc_outputs(plan)
    plan.run(**ins, **eager)
    assert plan.device_status() == 0
    outs = alloc_outputs(plan)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        plan.run(stream=stream, **ins, **outs)          # warm-up on the capture stream
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream=stream, **ins, **outs)
    for _ in range(2):
        for t in outs.values():
            t.fill_(0x33 if t.dtype == torch.uint8 else 7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        for k, t in outs.items():
            assert torch.equal(t, eager[k]), k
