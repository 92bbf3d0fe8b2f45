"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element
by element, on problems the oracle finishes in seconds: several tiles, ragged
groups (empty ones included), K and N tails, every epilogue and output format.

Tolerances: BF16/F16/F32 D within 2^-7 |ref| + 1e-3 rms(ref); FP8/FP4 D and
the scale factors bit-equal on >= 99.9% of elements and blocks, the rest
within one code step; amax within 2^-10 relative.
"""
import numpy as np
import pytest
import torch

from helpers import oracle_inputs, oracle_run, small_problem
from gpu_harness import TILES, tile_id, alloc_outputs, compare, make_plan, run_gpu, to_device, SENTINEL
from block_scaled_grouped_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _spread_scales(p, seed=7):
    g = torch.Generator().manual_seed(seed)
    lo, hi = (0x30, 0x40) if p.in_fmt == "nvfp4" else (122, 132)
    p.sfa_rows = torch.randint(lo, hi, p.sfa_rows.shape, generator=g).to(torch.uint8)
    p.sfb_rows = torch.randint(lo, hi, p.sfb_rows.shape, generator=g).to(torch.uint8)
    return p


def _parity(p, gate_first=False, check_amax=True, tile=(0, 0)):
    ref = oracle_run(p, gate_first=int(gate_first))
    outs, sfa, sfb = run_gpu(p, gate_first=gate_first, tile=tile)
    ins = oracle_inputs(p)
    # the library's packer and the oracle's index map agree byte for byte
    assert np.array_equal(sfa.cpu().numpy(), ins["sfa"])
    assert np.array_equal(sfb.cpu().numpy(), ins["sfb"])
    compare(p, outs, ref)
    if "amax" in outs and check_amax:
        got = outs["amax"].cpu().numpy()
        np.testing.assert_allclose(got, ref["amax"], rtol=2.0 ** -10, atol=0)
    return outs, ref


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_tiny_workload(tile):
    _parity(W.workload("tiny"), tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_gate_bf16_ragged_groups_and_k_tail(tile):
    # groups 300, 0, 129, 1000, 64 rows -> padded to 128; K=416 leaves a 32-column stage
    p = small_problem(counts=(300, 0, 129, 1000, 64), k=416, n=384, pad_to=128, seed=21)
    _parity(_spread_scales(p), tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_first_and_last_group_empty_and_n_tail(tile):
    p = small_problem(counts=(0, 200, 0, 130, 0), k=256, n=96, pad_to=128, seed=22)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_single_group_f32_and_f16(tile):
    p = small_problem(counts=(256,), k=512, n=256, pad_to=128, out_fmt="f32", seed=23)
    _parity(_spread_scales(p), tile=tile)
    # unit-range scales keep D inside F16's range (65504)
    p = small_problem(counts=(256,), k=512, n=256, pad_to=128, out_fmt="f16", seed=23)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_f16_overflow_reads_as_infinity(tile):
    """F16 D beyond the format's range is converted as IEEE round-to-nearest-
    even does: |D| >= 65520 (half-way to the next binade) becomes +-inf, no
    saturation.  The per-group amax is taken from the unrounded D, so it stays
    finite and matches the oracle's.  alpha = 2048 on the first group puts a
    part of its D above the range; the second group stays inside it."""
    p = small_problem(counts=(256, 100), k=512, n=256, pad_to=128, out_fmt="f16", seed=27,
                      alpha=[2048.0, 1.0])
    ref = oracle_run(p)
    outs, _, _ = run_gpu(p, tile=tile)
    from gpu_harness import decode_float_out, check_float_d
    d = decode_float_out(outs["d"].cpu().numpy(), "f16", p.m_pad, p.n_out)
    r = ref["d_ref"]
    over = np.abs(r) >= 65520.0 * (1 + 2.0 ** -7)
    inside = np.abs(r) <= 65504.0 * (1 - 2.0 ** -7)
    assert over.sum() > 100 and inside.sum() > 100, (over.sum(), inside.sum())
    assert np.all(np.isinf(d[over])) and np.all(np.sign(d[over]) == np.sign(r[over]))
    check_float_d(d[inside], r[inside])
    assert np.all(np.isfinite(outs["amax"].cpu().numpy()))
    np.testing.assert_allclose(outs["amax"].cpu().numpy(), ref["amax"], rtol=2.0 ** -10, atol=0)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_e5m2_inputs(tile):
    p = small_problem(counts=(128, 100), k=256, n=128, pad_to=128, in_fmt="mxfp8_e5m2", seed=24)
    _parity(p, tile=tile)


@pytest.mark.parametrize("gate_first", [False, True])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_swiglu_e4m3_row_and_col(gate_first, tile):
    p = small_problem(counts=(130, 256, 40), k=384, n=512, pad_to=128, epi="swiglu",
                      out_fmt="e4m3", want_col=True, seed=25)
    _parity(_spread_scales(p), gate_first=gate_first, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_srelu_clamp_e4m3_norm_half(tile):
    p = small_problem(counts=(200, 0, 77), k=256, n=256, pad_to=128, epi="srelu", out_fmt="e4m3",
                      want_col=True, tanh_clamp_s=8.0, norm_const=0.5, seed=26)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_srelu_e5m2_and_bf16(tile):
    p = small_problem(counts=(128, 300), k=512, n=256, pad_to=128, epi="srelu", out_fmt="e5m2",
                      want_col=True, seed=27)
    _parity(p, tile=tile)
    p = small_problem(counts=(128, 300), k=512, n=256, pad_to=128, epi="srelu", out_fmt="bf16",
                      tanh_clamp_s=4.0, seed=28)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_mxfp8_to_e2m1_with_columns(tile):
    p = small_problem(counts=(256, 90), k=256, n=256, pad_to=128, epi="gate", out_fmt="e2m1",
                      want_col=True, seed=29)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_gate_bf16(tile):
    p = small_problem(counts=(150, 0, 300), k=512, n=384, pad_to=128, in_fmt="nvfp4", seed=30)
    _parity(_spread_scales(p), tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_k_tail(tile):
    # K = 288: the last stage holds 32 FP4 elements (one MMA of 64, half zero-filled)
    p = small_problem(counts=(128, 128), k=288, n=128, pad_to=128, in_fmt="nvfp4", seed=31)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_srelu_clamp_e2m1(tile):
    p = small_problem(counts=(300, 128, 0, 50), k=512, n=256, pad_to=128, in_fmt="nvfp4",
                      epi="srelu", out_fmt="e2m1", tanh_clamp_s=8.0, seed=32)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_e2m1_row_and_16_row_column_blocks(tile):
    # NVFP4 inputs: E4M3 scales per 16 values for D rows and for D_col columns
    p = small_problem(counts=(256, 70, 0, 130), k=512, n=256, pad_to=128, in_fmt="nvfp4",
                      epi="gate", out_fmt="e2m1", want_col=True, seed=36)
    _parity(p, tile=tile)
    p = small_problem(counts=(128, 200), k=256, n=256, pad_to=128, in_fmt="nvfp4",
                      epi="srelu", out_fmt="e2m1", want_col=True, tanh_clamp_s=4.0, seed=37)
    _parity(p, tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_nvfp4_swiglu_bf16(tile):
    p = small_problem(counts=(128, 200), k=256, n=256, pad_to=128, in_fmt="nvfp4",
                      epi="swiglu", out_fmt="bf16", seed=33)
    _parity(p, tile=tile)


def _sparse_counts(num_groups, filled, seed):
    """num_groups groups, all empty except `filled` ones (first, last and
    random ones), each 1..300 rows."""
    rng = np.random.default_rng(seed)
    counts = [0] * num_groups
    idx = {0, num_groups - 1} | set(int(i) for i in rng.choice(num_groups, filled - 2, replace=False))
    for i in idx:
        counts[i] = int(rng.integers(1, 301))
    return counts


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_1024_groups_mostly_empty(tile):
    # the largest expert count the pages allow (L <= 1024), 14 groups non-empty
    p = small_problem(counts=_sparse_counts(1024, 14, seed=40), k=128, n=256, pad_to=128, seed=40)
    _parity(_spread_scales(p), tile=tile)


@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_1024_groups_nvfp4_e2m1(tile):
    p = small_problem(counts=_sparse_counts(1024, 10, seed=41), k=256, n=256, pad_to=128,
                      in_fmt="nvfp4", epi="srelu", out_fmt="e2m1", want_col=True, seed=41)
    _parity(p, tile=tile)


def test_bad_offsets_are_reported_and_nothing_is_written():
    p = to_device(small_problem(counts=(128, 128), k=128, n=128, pad_to=128, seed=34))
    for bad in ([100, 256], [256, 128], [128, 384]):
        p.padded_offsets = torch.tensor(bad, dtype=torch.int32, device="cuda")
        plan = make_plan(p)
        outs = alloc_outputs(plan)
        import block_scaled_grouped_gb300 as bsgg
        norm = torch.ones(1, device="cuda")
        plan.run(a=p.a, sfa=bsgg.pack_sf(p.sfa_rows), b=p.b, sfb=bsgg.pack_sf(p.sfb_rows),
                 padded_offsets=p.padded_offsets, alpha=p.alpha, prob=p.prob, norm_const=norm, **outs)
        assert plan.device_status() == 5
        assert (outs["d"] == SENTINEL).all()


@pytest.mark.parametrize("size", ["small", "large"])
def test_host_buffer_call_matches_device_call(size):
    """bsgg_run_host against bsgg_run on the same inputs, bit for bit, on a small
    problem and on one whose A, B, D and D_col copies are several MB each."""
    if size == "small":
        p = small_problem(counts=(200, 60), k=256, n=256, pad_to=128, epi="swiglu", out_fmt="e4m3",
                          want_col=True, seed=35)
    else:
        p = small_problem(counts=(1500, 700), k=2048, n=4096, pad_to=128, epi="swiglu", out_fmt="e4m3",
                          want_col=True, seed=36)
        assert p.a.numel() >= 4 << 20 and p.m_pad * p.n // 2 >= 4 << 20
    pd = to_device(p)
    outs, sfa, sfb = run_gpu(pd)
    plan = make_plan(pd)
    dev = alloc_outputs(plan)
    dev.update(a=torch.empty_like(pd.a), sfa=torch.empty_like(sfa), b=torch.empty_like(pd.b),
               sfb=torch.empty_like(sfb), padded_offsets=torch.empty_like(pd.padded_offsets),
               alpha=torch.empty_like(pd.alpha), prob=torch.empty_like(pd.prob),
               norm_const=torch.empty(1, device="cuda"))
    host = dict(a=p.a.pin_memory(), sfa=sfa.cpu().pin_memory(), b=p.b.pin_memory(),
                sfb=sfb.cpu().pin_memory(), padded_offsets=p.padded_offsets.pin_memory(),
                alpha=p.alpha.pin_memory(), prob=p.prob.pin_memory(),
                norm_const=torch.tensor([p.norm_const]).pin_memory())
    for k_, t in outs.items():
        host[k_] = torch.empty(t.shape, dtype=t.dtype).pin_memory()
    h2d, d2h = plan.run_host(host, dev)
    assert h2d == sum(host[k_].numel() * host[k_].element_size() for k_ in
                      ("a", "sfa", "b", "sfb", "padded_offsets", "alpha", "prob", "norm_const"))
    assert d2h == sum(t.numel() * t.element_size() for t in outs.values())
    for k_, t in outs.items():
        assert torch.equal(host[k_], t.cpu()), k_


def test_async_host_calls_in_flight_on_two_streams():
    """bsgg_run_host_async: four batches (the same A, different routing
    probabilities), two in flight at a time on two streams, each stream with
    its own plan, device buffers and host output buffers; every batch's
    outputs equal bsgg_run's on its inputs, bit for bit."""
    import dataclasses
    p = small_problem(counts=(300, 200), k=512, n=512, pad_to=128, epi="swiglu", out_fmt="e4m3",
                      want_col=True, seed=40)
    pd = to_device(p)
    probs = [p.prob * f for f in (1.0, 0.5, 2.0, 0.25)]
    refs = []
    for pr in probs:
        outs, sfa, sfb = run_gpu(dataclasses.replace(pd, prob=pr.cuda()))
        refs.append({k_: t.cpu() for k_, t in outs.items()})
    streams = [torch.cuda.Stream() for _ in range(2)]
    plans = [make_plan(pd) for _ in range(2)]
    devs = []
    for plan in plans:
        dev = alloc_outputs(plan)
        dev.update(a=torch.empty_like(pd.a), sfa=torch.empty_like(sfa), b=pd.b, sfb=sfb,
                   padded_offsets=pd.padded_offsets, alpha=pd.alpha, prob=torch.empty_like(pd.prob),
                   norm_const=torch.tensor([p.norm_const], device="cuda"))
        devs.append(dev)
    host_in = dict(a=p.a.pin_memory(), sfa=sfa.cpu().pin_memory())
    host_outs = [{k_: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k_, t in refs[0].items()}
                 for _ in probs]
    host_probs = [pr.pin_memory() for pr in probs]   # alive until the copies have run
    torch.cuda.synchronize()
    for i, pr in enumerate(host_probs):
        j = i % 2
        host = dict(host_in, prob=pr, **host_outs[i])
        h2d, d2h = plans[j].run_host(host, devs[j], stream=streams[j], sync=False)
        assert h2d == sum(host[k_].numel() * host[k_].element_size() for k_ in ("a", "sfa", "prob"))
    torch.cuda.synchronize()
    for j in range(2):
        assert plans[j].device_status(streams[j]) == 0
    for i in range(len(probs)):
        for k_, t in refs[i].items():
            assert torch.equal(host_outs[i][k_], t), (i, k_)


@pytest.mark.parametrize("in_fmt", ["fp4_ue8m0_16", "mxfp4"])
@pytest.mark.parametrize("tile", TILES, ids=tile_id)
def test_fp4_with_ue8m0_scales(tile, in_fmt):
    """FP4 data with UE8M0 scales per 16 or 32 (the Quant page's NVF4 rows with
    float8_e8m0fnu scales): BF16 gate and E2M1 sReLU outputs (UE8M0 output
    scales of the input's block length), ragged groups and a K tail, spread
    scales."""
    p = small_problem(counts=(150, 0, 300), k=544, n=384, pad_to=128, in_fmt=in_fmt, seed=38)
    _parity(_spread_scales(p), tile=tile)
    p = small_problem(counts=(256, 70, 0, 130), k=512, n=256, pad_to=128, in_fmt=in_fmt, epi="srelu",
                      out_fmt="e2m1", want_col=True, tanh_clamp_s=8.0, seed=39)
    _parity(p, tile=tile)
