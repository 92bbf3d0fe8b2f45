"""Benchmark of the grouped block-scaled GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
                    [--workload fc1_swiglu|fc2_gate|fine_nvfp4|skewed|fc1_dswiglu|fc1_dswiglu_bf16|skinny|tiny]

A step is one bsgg_run over one batch of the workload (all of the hot path:
scheduling, operand fetch, block-scaled MMA, alpha/prob, activation,
quantization, stores).  The default workload is MoE FC1 + SwiGLU (4096 tokens
top-2 over 8 experts, K=4096, N=28672, MXFP8 in, E4M3 D and D_col with UE8M0
SFD_row/SFD_col).  Inputs are seeded synthetic tensors generated on the device
before timing; they are larger than L2, and steps run back to back.

Metric: TFLOP/s of 2 * valid_rows * N * K (padding rows excluded).  The JSON
line also carries the roofline of the kernel (against the measured bf16 peak
scaled to the dtype by the nominal dense ratio, and against this GPU's measured
block-scaled MMA rate of the instruction form the launch issues), the
end-to-end number through the host-buffer C-ABI call, the CPU oracle baseline,
and the SM clocks sampled during the timed region.  After the headline
workload the default run times every other hot-path workload (FC2 gated,
fine-grained NVFP4, skewed, skinny, tiny) the same way, --extra-steps steps
each, under the line's "workloads" key.

N > 1 (torchrun): every rank runs an independent replica on its own GPU (the
operation has no exchange step); value = all ranks' FLOPs / max rank time.
--impl reference times the CPU oracle (rank 0 only) on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped GEMM TFLOP/s (valid rows) and % of GB300 dense FP8/FP4 peak, 1 GPU"
UNIT = "TFLOP/s"
# nominal dense tensor throughput relative to bf16 (2.25 PFLOP/s): fp8 4.5, fp4 13.5
DTYPE_RATIO = {"mxfp8_e4m3": 2.0, "mxfp8_e5m2": 2.0, "nvfp4": 6.0, "fp4_ue8m0_16": 6.0, "mxfp4": 6.0, "bf16": 1.0}
DTYPE_NAME = {"mxfp8_e4m3": "mxfp8(e4m3,ue8m0/32)", "mxfp8_e5m2": "mxfp8(e5m2,ue8m0/32)",
              "nvfp4": "nvfp4(e2m1,e4m3/16)", "fp4_ue8m0_16": "fp4(e2m1,ue8m0/16)", "mxfp4": "mxfp4(e2m1,ue8m0/32)",
              "bf16": "bf16"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the sources that make up bsgg_kernel and its launch (not the
    peak-measurement unit)."""
    d = os.path.join(ROOT, "block_scaled_grouped_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name == "bsgg_peak.cu":
            continue
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, mx, reasons, power = [], [], set(), []
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
                power.append(float(f[4]))
            except ValueError:
                continue
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if f[col].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:   # CPU ranks (tests of the multi-rank logic)
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_inputs(p):
    """Host copies of a problem's inputs with the oracle's own scale packing."""
    import oracle as orc
    np_ = lambda t: t.detach().cpu().contiguous().numpy()
    ins = dict(a=np_(p.a), b=np_(p.b), sfa=orc.pack_sf(np_(p.sfa_rows)), sfb=orc.pack_sf(np_(p.sfb_rows)),
               padded_offsets=np_(p.padded_offsets), alpha=np_(p.alpha), prob=np_(p.prob))
    if p.saved_c is not None:
        ins.update(saved_c=np_(p.saved_c.double()), beta=np_(p.beta))
    return ins


def oracle_sample(p, ins, budget_s: float, max_blocks: int = 64, seed: int = 0):
    """Time the oracle on 32-row blocks of real rows, one call per block, until
    budget_s of wall time is spent.  Returns (flops, seconds, blocks, threads)."""
    import oracle as orc
    code_in = {"mxfp8_e4m3": orc.IN_MXFP8_E4M3, "mxfp8_e5m2": orc.IN_MXFP8_E5M2, "nvfp4": orc.IN_NVFP4,
               "fp4_ue8m0_16": orc.IN_FP4_UE8M0_16, "mxfp4": orc.IN_MXFP4, "bf16": orc.IN_BF16}
    code_out = {"bf16": orc.OUT_BF16, "f16": orc.OUT_F16, "f32": orc.OUT_F32, "e4m3": orc.OUT_E4M3,
                "e5m2": orc.OUT_E5M2, "e2m1": orc.OUT_E2M1}
    code_epi = {"gate": orc.EPI_GATE, "swiglu": orc.EPI_SWIGLU, "srelu": orc.EPI_SRELU, "geglu": orc.EPI_GEGLU,
                "dswiglu": orc.EPI_DSWIGLU, "dgeglu": orc.EPI_DGEGLU, "dsituglu": orc.EPI_DSITUGLU}
    off = ins["padded_offsets"]
    starts = np.concatenate([[0], off[:-1]])
    real_blocks = np.unique(np.concatenate(
        [np.arange(s, s + c) // 32 for s, c in zip(starts, p.counts) if c > 0]))
    rng = np.random.default_rng(seed)
    order = rng.permutation(real_blocks)[:max_blocks]
    threads = os.cpu_count() or 1
    done, t0 = [], time.perf_counter()
    for b in order:
        orc.run(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_fmt=code_in[p.in_fmt],
                out_fmt=code_out[p.out_fmt], epi=code_epi[p.epi], norm_const=p.norm_const,
                tanh_clamp_s=p.tanh_clamp_s, want_col=p.want_col, blocks=np.array([b]),
                threads=threads, **ins)
        done.append(int(b))
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    real = np.zeros(p.m_pad, dtype=bool)
    for st_, c in zip(starts, p.counts):
        real[st_:st_ + c] = True
    rows_real = int(sum(real[32 * b:32 * b + 32].sum() for b in done))
    flops = 2.0 * rows_real * p.n * p.k
    return flops, secs, done, threads


def make_workload(name: str, device):
    from block_scaled_grouped_gb300 import workloads as W
    return W.workload(name, device=device)


def algorithmic_bytes(p) -> int:
    """Bytes a launch must move at least: A, SFA, the B and SFB slices of the
    non-empty groups, and the outputs (D, D_col, SFD_row, SFD_col or amax);
    for the backward epilogues also the saved C read and dprob written."""
    from block_scaled_grouped_gb300 import workloads as W
    def cdiv(a, b):
        return -(-a // b)

    def sfb(rows, cols, v, slices=1):
        return 512 * slices * cdiv(rows, 128) * cdiv(cdiv(cols, v), 4)
    fp4 = p.in_fmt in ("nvfp4", "fp4_ue8m0_16", "mxfp4")
    v = p.sf_vec
    kb = p.k // 2 if fp4 else 2 * p.k if p.in_fmt == "bf16" else p.k
    ks = 0 if p.in_fmt == "bf16" else p.k      # bf16 operands have no scale factors
    off = [int(x) for x in p.padded_offsets.tolist()]
    nonempty = sum(1 for g, e in enumerate(off) if e > (off[g - 1] if g else 0))
    n_out = p.n_out
    bits = {"bf16": 16, "f16": 16, "f32": 32, "e4m3": 8, "e5m2": 8, "e2m1": 4}[p.out_fmt]
    d = p.m_pad * n_out * bits // 8
    out = d * (2 if p.want_col else 1)
    if p.out_fmt in ("e4m3", "e5m2", "e2m1"):
        out += sfb(p.m_pad, n_out, v) + (sfb(n_out, p.m_pad, v) if p.want_col else 0)
    else:
        out += 4 * p.num_groups * (2 if p.epi in W.BWD_EPILOGUES else 1)
    extra = 0
    if p.epi in W.BWD_EPILOGUES:
        extra = p.saved_c.numel() * p.saved_c.element_size() + 4 * p.m_pad + 4 * p.num_groups
    return (p.m_pad * kb + sfb(p.m_pad, ks, v) + nonempty * p.n * kb + sfb(p.n, ks, v, nonempty) + out
            + extra)


def roofline_bound(flops: float, alg_bytes: float, peak_tflops: float, peak_gbs: float) -> str:
    """"tensor" when the launch's arithmetic intensity (valid FLOPs per
    algorithmic byte) reaches the ridge point of the two peaks, else "hbm"."""
    return "tensor" if flops / alg_bytes >= (peak_tflops * 1e12) / (peak_gbs * 1e9) else "hbm"


def config_of(p, extra=None):
    c = {"workload": p.name, "experts": p.num_groups, "rows_valid": p.m_real, "rows_padded": p.m_pad,
         "n": p.n, "k": p.k, "in": DTYPE_NAME[p.in_fmt], "out": p.out_fmt, "epilogue": p.epi,
         "tanh_clamp_s": p.tanh_clamp_s or None, "col_outputs": p.want_col, "norm_const": p.norm_const,
         "l2": "inputs larger than L2 (no flush between steps)"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    device = "cuda" if torch.cuda.is_available() else "cpu"
    p = make_workload(args.workload, device)
    per_step_budget = args.ref_step_seconds
    import oracle
    oracle.build()
    ins = oracle_inputs(p)
    for _ in range(args.warmup):
        oracle_sample(p, ins, 0.0, max_blocks=1, seed=1000 + _)
    tot_f, tot_s, blocks_all, threads = 0.0, 0.0, [], 1
    for s in range(args.steps):
        f, sec, blocks, threads = oracle_sample(p, ins, per_step_budget, max_blocks=1, seed=s)
        tot_f += f
        tot_s += sec
        blocks_all += blocks
    value = tot_f / tot_s / 1e12
    sample = (f"{len(blocks_all)} 32-row blocks of valid rows (all N={p.n} columns, K={p.k}), "
              f"one per step; fp64 oracle, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config_of(p, {"parallelism": "none (CPU oracle)"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def mma_form(p, tile_arg: str):
    """(tile_m, tile_n) of the MMA instruction form a launch of p issues: the
    --tile given, else the library's default (CTA pairs, 256 x 256, except
    128 x 128 single CTAs for the block-scaled backward epilogues)."""
    if tile_arg:
        tm, tn = (int(x) for x in tile_arg.split("x"))
        return tm, tn
    from block_scaled_grouped_gb300 import workloads as W
    if p.epi in W.BWD_EPILOGUES and p.in_fmt != "bf16":
        return 128, 128
    return 256, 256


_MMA_PEAK_CACHE = {}


def measured_mma_peak(in_fmt: str, form):
    """The block-scaled MMA rate of this GPU for the dtype and instruction form
    (bsgg_measure_mma_peak_tile: operands resident in shared memory, no loads,
    no epilogue), best of three, with the SM clock sampled meanwhile; None for
    bfloat16 operands (no block-scaled form)."""
    import block_scaled_grouped_gb300 as bsgg
    probe = {"mxfp8_e4m3": "mxfp8_e4m3", "mxfp8_e5m2": "mxfp8_e4m3", "nvfp4": "nvfp4",
             "fp4_ue8m0_16": "nvfp4", "mxfp4": "nvfp4"}.get(in_fmt)
    if probe is None:
        return None
    key = (probe, tuple(form))
    if key not in _MMA_PEAK_CACHE:
        tm, tn = form
        bsgg.measure_mma_peak_tile(probe, tm, tn, 1 << 16)          # warm-up
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        sampler.mark(True)
        v = max(bsgg.measure_mma_peak_tile(probe, tm, tn, 1 << 21) for _ in range(3))
        sampler.mark(False)
        clocks = sampler.stop()
        _MMA_PEAK_CACHE[key] = {"value": v, "unit": UNIT,
                                "form": f"cta_group::{2 if tm == 256 else 1} M={tm} N={tn} "
                                        f"({'kind::mxf4nvf4 K=64' if probe == 'nvfp4' else 'kind::mxf8f6f4 K=32'})",
                                "sm_mhz": clocks.get("sm_mhz"), "reasons": clocks.get("reasons")}
    return _MMA_PEAK_CACHE[key]


L2_FLUSH_BYTES = 512 << 20           # four times the 129 MB L2


def time_l2_cold(p, plan, tensors, stream, dev, steps: int) -> dict:
    """Each launch after a write of L2_FLUSH_BYTES to a scratch buffer (so that
    no input or output line stays in L2 from the previous step), timed alone
    with CUDA events on the launching stream; the writes fall outside the
    events."""
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for e0, e1 in evs:
        scratch.fill_(1)
        e0.record(stream)
        plan.run(stream=stream, **tensors)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if plan.device_status(stream) != 0:
        raise RuntimeError(f"device status after the L2-cold steps ({p.name})")
    ms = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
    mean = sum(ms) / len(ms)
    del scratch
    return {"value": p.flops / (mean * 1e-3) / 1e12, "unit": UNIT, "steps": steps, "ms_per_step": mean,
            "median_ms": ms[len(ms) // 2], "flush_bytes": L2_FLUSH_BYTES,
            "what": "each launch timed alone (CUDA events) after a write of flush_bytes evicted L2"}


def make_plan(p, args):
    """The plan of workload `p` in the tile shape and cluster `args` ask for."""
    import block_scaled_grouped_gb300 as bsgg
    tile = tuple(int(x) for x in args.tile.split("x")) if args.tile else (0, 0)
    cluster = tuple(int(x) for x in args.cluster.split("x")) if args.cluster else (0, 0)
    return bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col,
                     tanh_clamp_s=p.tanh_clamp_s, tile=tile, cluster=cluster)


def time_workload(p, args, dev, world, steps: int, warmup: int):
    """Times `steps` back-to-back runs of one workload's launch after `warmup`
    untimed ones (CUDA events on the launching stream, a barrier and a device
    synchronize on both sides, SM clocks sampled meanwhile).  Returns the
    record (value, ms_per_step, roofline, hbm, clocks, ...), the plan and the
    tensors."""
    import block_scaled_grouped_gb300 as bsgg
    plan = make_plan(p, args)
    sfa = bsgg.pack_sf(p.sfa_rows)
    sfb = bsgg.pack_sf(p.sfb_rows)
    outs = {}
    for name, nbytes in plan.output_bytes().items():
        if name == "amax":
            outs[name] = torch.zeros(nbytes // 4, dtype=torch.float32, device=dev)
        else:
            outs[name] = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device=dev)
    tensors = dict(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha,
                   prob=p.prob, norm_const=norm, **outs)
    if p.saved_c is not None:
        # the backward's saved C and beta, and dprob (accumulated across steps:
        # the timing does not depend on its values)
        tensors.update(saved_c=p.saved_c, beta=p.beta,
                       dprob=torch.zeros(p.m_pad, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)

    for _ in range(warmup):
        plan.run(stream=stream, **tensors)
    st = plan.device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up ({p.name})")

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.mark(True)
    ev0.record(stream)
    for _ in range(steps):
        plan.run(stream=stream, **tensors)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(False)
    barrier(world)
    clocks = sampler.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    st = plan.device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region ({p.name})")
    t_max_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = t_max_ms / steps
    value = world * steps * p.flops / (t_max_ms * 1e-3) / 1e12

    # roofline of the (single) kernel of a step
    peaks, peak_kind = measured_peaks()
    ratio = DTYPE_RATIO[p.in_fmt]
    peak = peaks["bf16_tflops"] * ratio
    achieved = p.flops / (elapsed_ms / steps * 1e-3) / 1e12
    # the recorded counters are of the library's default tile shape
    traffic = recorded_traffic(p.name) if not (args.tile or args.cluster) else None
    alg_bytes = algorithmic_bytes(p)
    hbm_gbs = alg_bytes / (elapsed_ms / steps * 1e-3) / 1e9
    bound = roofline_bound(p.flops, alg_bytes, peak, peaks["hbm_gbs"])
    hbm = {"algorithmic_bytes": alg_bytes, "achieved_gbs": hbm_gbs, "peak_gbs": peaks["hbm_gbs"],
           "frac": hbm_gbs / peaks["hbm_gbs"],
           "what": "algorithmic bytes per launch / kernel time" + (
               " (not the bound of this kernel)" if bound == "tensor" else " (the bound of this kernel)")}
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": (f"{peak_kind} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                                f"{ratio:g} (nominal dense {DTYPE_NAME[p.in_fmt]}/bf16 ratio)"),
                "kernel": "bsgg_kernel", "flops_per_launch": p.flops,
                "flops_incl_padding": 2.0 * p.m_pad * p.n * p.k}
    # the stricter denominator: this GPU's measured rate of the instruction form
    # the launch issues
    mma = None if args.no_mma_peak else measured_mma_peak(p.in_fmt, mma_form(p, args.tile))
    if mma is not None:
        roofline["measured_mma_peak"] = mma
        roofline["frac_of_measured_mma"] = achieved / mma["value"]
    if bound == "hbm":
        # below the ridge point (few rows per expert): the bound is the bytes
        roofline.update({"bound": "hbm", "achieved": hbm_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": hbm_gbs / peaks["hbm_gbs"],
                         "peak_source": f"{peak_kind} HBM copy bandwidth {peaks['hbm_gbs']} GB/s",
                         "bytes_per_launch": alg_bytes, "tflops": achieved})
    rec = {"value": value, "unit": UNIT, "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
           "elapsed_ms": elapsed_ms, "clocks": clocks, "roofline": roofline, "hbm": hbm,
           "pct_of_dtype_peak": 100.0 * achieved / peak, "config": config_of(p),
           "gpu_launches": steps * plan.launches_per_run}
    return rec, plan, tensors


# the other workloads the default run also times (every hot-path config and the
# decode-like skinny case), after the headline
EXTRA_WORKLOADS = ("fc2_gate", "fine_nvfp4", "skewed", "skinny", "tiny")


def run_gpu(args, world, rank, local):
    import block_scaled_grouped_gb300 as bsgg
    from block_scaled_grouped_gb300 import build as bsgg_build
    bsgg_build.build()
    dev = torch.device("cuda", local if world > 1 else 0)
    t0 = time.time()
    p = make_workload(args.workload, dev)
    torch.cuda.synchronize()
    log(f"[bench] workload {p.name}: m_pad={p.m_pad} valid={p.m_real} n={p.n} k={p.k} "
        f"generated in {time.time() - t0:.1f}s")
    rec, plan, tensors = time_workload(p, args, dev, world, args.steps, args.warmup)
    stream = torch.cuda.current_stream(dev)
    # the same launches with L2 evicted before each (the main timing relies on
    # inputs larger than L2 instead)
    l2_cold = time_l2_cold(p, plan, tensors, stream, dev, min(args.steps, 20))

    # end to end through the host-buffer C-ABI call.  Headline: an MoE layer's
    # step -- the expert weights (B, SFB) and alpha stay resident in HBM, the
    # step's activations (A, SFA), routing (padded_offsets, prob) and norm_const
    # are copied in from pinned host memory and every output is copied back.
    # Also reported: the same with the weights copied in every step as well.
    e2e = None
    if not args.no_e2e:
        host = {}
        for k_, t in tensors.items():
            host[k_] = torch.empty(t.shape, dtype=t.dtype).pin_memory()
        for k_ in ("a", "sfa", "b", "sfb", "padded_offsets", "alpha", "prob", "norm_const", "saved_c",
                   "beta", "dprob"):
            if k_ in tensors:
                host[k_].copy_(tensors[k_].cpu())
        dev_bufs = dict(tensors)
        resident = ("b", "sfb", "alpha", "beta")
        host_layer = {k_: v for k_, v in host.items() if k_ not in resident}
        n_e2e = max(3, min(args.steps, 10))

        def timed(h):
            plan.run_host(h, dev_bufs, stream=stream)      # warm-up
            torch.cuda.synchronize(dev)
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                nb = plan.run_host(h, dev_bufs, stream=stream)
            return max_over_ranks((time.perf_counter() - t0) / n_e2e, world), nb

        # two steps in flight: bsgg_run_host_async on two streams, each with its
        # own plan, device buffers for everything copied, and host output
        # buffers, so that one step's outputs travel to the host while the next
        # step's inputs travel in and its kernel runs; every step's copies are
        # inside the timed region, which ends when both streams have finished
        plan2 = make_plan(p, args)
        dev2 = {k_: (v if k_ in resident else torch.empty_like(v)) for k_, v in dev_bufs.items()}
        # (the backward's dprob is copied in and out: the second stream gets
        # its own host buffer, whose values do not affect the timing)
        outputs = [k_ for k_ in host_layer if k_ not in ("a", "sfa", "padded_offsets", "prob", "norm_const",
                                                        "saved_c")]
        host2 = dict(host_layer, **{k_: torch.empty_like(host_layer[k_]).pin_memory() for k_ in outputs})
        streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        lanes = [(plan, dev_bufs, host_layer), (plan2, dev2, host2)]

        def timed_pipelined():
            for j, (pl, dv, hs) in enumerate(lanes):         # warm-up
                pl.run_host(hs, dv, stream=streams[j], sync=False)
            torch.cuda.synchronize(dev)
            barrier(world)
            t0 = time.perf_counter()
            for i in range(2 * n_e2e):
                pl, dv, hs = lanes[i % 2]
                nb = pl.run_host(hs, dv, stream=streams[i % 2], sync=False)
            torch.cuda.synchronize(dev)
            return max_over_ranks((time.perf_counter() - t0) / (2 * n_e2e), world), nb
        pipe_s, (h2d, d2h) = timed_pipelined()
        for j, (pl, _, _) in enumerate(lanes):
            if pl.device_status(streams[j]) != 0:
                raise RuntimeError(f"device status after the end-to-end steps ({p.name})")
        plan2.close()
        sync_s, _ = timed(host_layer)
        all_s, (h2d_all, d2h_all) = timed(host)
        e2e = {"value": world * p.flops / pipe_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": pipe_s * 1e3,
               "what": "bsgg_run_host_async per step, two steps in flight on two streams: A, SFA, "
                       "padded_offsets, prob, norm_const copied in from pinned host memory, every "
                       "output copied back to pinned host memory, both streams synchronized at the "
                       "end; expert weights B, SFB and alpha resident in HBM",
               "synchronous": {"value": world * p.flops / sync_s / 1e12, "unit": UNIT,
                               "ms_per_step": sync_s * 1e3,
                               "what": "bsgg_run_host per step, the stream synchronized after each"},
               "all_inputs_copied": {"value": world * p.flops / all_s / 1e12, "unit": UNIT,
                                     "h2d_bytes_per_step": h2d_all, "d2h_bytes_per_step": d2h_all,
                                     "ms_per_step": all_s * 1e3,
                                     "what": "bsgg_run_host per step with B, SFB and alpha copied in too"}}
        del host, host_layer, host2, dev_bufs, dev2
    plan.close()
    gpu_launches = rec["gpu_launches"]
    del tensors

    # every other workload of the hot path, each timed the same way (its own
    # warm-up, extra_steps steps), its tensors freed before the next one
    workloads = {}
    if not args.no_extra_workloads:
        for name in EXTRA_WORKLOADS:
            if name == p.name:
                continue
            t0 = time.time()
            q = make_workload(name, dev)
            torch.cuda.synchronize(dev)
            log(f"[bench] workload {q.name}: m_pad={q.m_pad} valid={q.m_real} generated in "
                f"{time.time() - t0:.1f}s")
            r, qplan, qt = time_workload(q, args, dev, world, args.extra_steps, args.warmup)
            qplan.close()
            del qt, q
            torch.cuda.empty_cache()
            gpu_launches += r["gpu_launches"]
            workloads[name] = {k_: r[k_] for k_ in ("value", "unit", "steps", "ms_per_step", "roofline",
                                                    "hbm", "clocks", "pct_of_dtype_peak", "config")}

    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        f, secs, blocks, threads = oracle_sample(p, oracle_inputs(p), args.cpu_seconds)
        cpu_baseline = {"value": f / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                        "sample": f"{len(blocks)} random 32-row blocks of valid rows, all N={p.n} "
                                  f"columns, K={p.k}; {secs:.1f} s of fp64 oracle work on "
                                  f"{threads} threads"}

    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[p.in_fmt],
                "data": "synthetic (seeded MoE routing, N(0,1) draws quantized to the input format)",
                "config": config_of(p, {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                        "tile": args.tile or "library default",
                                        "cluster": args.cluster or "library default"}),
                "gpu_launches": gpu_launches, "clocks": rec["clocks"], "roofline": rec["roofline"],
                "e2e": e2e, "cpu_baseline": cpu_baseline, "hbm": rec["hbm"], "l2_cold": l2_cold,
                "pct_of_dtype_peak": rec["pct_of_dtype_peak"]}
        if workloads:
            line["workloads"] = workloads
        print(json.dumps(line), flush=True)


def run_mma_peak():
    """The tensor pipe's dense block-scaled rate on resident operands, with the
    SM clock sampled meanwhile."""
    import block_scaled_grouped_gb300 as bsgg
    from block_scaled_grouped_gb300 import build as bsgg_build
    bsgg_build.build()
    sampler = ClockSampler(0)
    res = {}
    forms = ((128, 128), (128, 256), (256, 256))      # cta_group::1 M=128; cta_group::2 M=256
    for fmt in ("mxfp8_e4m3", "nvfp4"):
        for tm, tn in forms:
            bsgg.measure_mma_peak_tile(fmt, tm, tn, 40000)          # warm-up
    sampler.start()
    sampler.mark(True)
    for fmt in ("mxfp8_e4m3", "nvfp4"):
        for tm, tn in forms:
            grp = 2 if tm == 256 else 1
            res[f"{DTYPE_NAME[fmt]} cta_group::{grp} M={tm} N={tn}"] = max(
                bsgg.measure_mma_peak_tile(fmt, tm, tn, 1 << 22) for _ in range(3))
    sampler.mark(False)
    clocks = sampler.stop()
    print(json.dumps({"metric": "dense block-scaled MMA TFLOP/s, operands resident in shared memory",
                      "unit": "TFLOP/s", "values": res, "clocks": clocks}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gpu", "reference"), default="gpu")
    ap.add_argument("--workload", default="fc1_swiglu")
    ap.add_argument("--tile", default="", help="MxN tile shape: 128x128, 128x256 or 256x256 "
                    "(a CTA pair); default: the library's choice")
    ap.add_argument("--cluster", default="", help="MxN cluster shape: 1x1 (128-row tiles) or 2x1 "
                    "(256x256 tiles on a CTA pair); default: the library's choice")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only --workload (by default the other hot-path workloads follow it)")
    ap.add_argument("--extra-steps", type=int, default=20, help="timed steps of each other workload")
    ap.add_argument("--no-mma-peak", action="store_true",
                    help="skip the MMA-rate measurement behind roofline.frac_of_measured_mma")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.0)
    ap.add_argument("--mma-peak", action="store_true", help="print the measured dense block-scaled "
                    "MMA throughput (bsgg_measure_mma_peak) for MXFP8 and NVFP4 and exit")
    args = ap.parse_args()
    if args.mma_peak:
        run_mma_peak()
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --impl gpu needs a CUDA device")
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
