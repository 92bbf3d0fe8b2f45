"""The benchmark's roofline arithmetic on CPU: which bound each workload's
launch meets (its valid FLOPs per algorithmic byte against the ridge point of
the dtype's peak and the HBM peak), and the decode-like "skinny" workload's
routing.  The workloads' shapes are taken from their routings alone (no
operand tensors are generated)."""
import types

import numpy as np
import pytest
import torch

import bench
from block_scaled_grouped_gb300 import workloads as W

PEAKS = {"hbm_gbs": 6777.6, "bf16_tflops": 1861.9}


def _meta(name, counts, k, n, in_fmt, out_fmt, epi, want_col):
    """The fields of a workloads.Problem that bench.algorithmic_bytes reads."""
    counts = np.asarray(counts, dtype=np.int64)
    padded = -(-counts // 128) * 128
    return types.SimpleNamespace(
        name=name, in_fmt=in_fmt, out_fmt=out_fmt, epi=epi, k=k, n=n,
        n_out=n // 2 if epi in ("swiglu", "geglu") else n,
        sf_vec=16 if in_fmt in ("nvfp4", "fp4_ue8m0_16") else 32,
        padded_offsets=torch.tensor(np.cumsum(padded), dtype=torch.int32),
        m_pad=int(padded.sum()), want_col=want_col, num_groups=int(counts.size),
        flops=2.0 * int(counts.sum()) * n * k, saved_c=None)


def _bound(p):
    peak = PEAKS["bf16_tflops"] * bench.DTYPE_RATIO[p.in_fmt]
    return bench.roofline_bound(p.flops, bench.algorithmic_bytes(p), peak, PEAKS["hbm_gbs"])


def _fc_counts():
    tokens, _ = W.route_softmax_topk(4096, 8, 2, seed=1)
    return [t.size for t in tokens]


def test_ridge_point():
    # ridge of 3723.8 TFLOP/s over 6777.6 GB/s: about 549 FLOP per byte
    assert bench.roofline_bound(550.0, 1.0, 3723.8, 6777.6) == "tensor"
    assert bench.roofline_bound(548.0, 1.0, 3723.8, 6777.6) == "hbm"


@pytest.mark.parametrize("name,meta,bound", [
    ("fc1_swiglu", lambda: _meta("fc1_swiglu", _fc_counts(), 4096, 28672, "mxfp8_e4m3", "e4m3", "swiglu", True),
     "tensor"),
    ("fc2_gate", lambda: _meta("fc2_gate", _fc_counts(), 14336, 4096, "mxfp8_e4m3", "bf16", "gate", False),
     "tensor"),
    ("fine_nvfp4", lambda: _meta("fine_nvfp4", [t.size for t in W.route_zipf_gumbel_topk(8192, 64, 8, 1.2, 4, 3)],
                                 7168, 2048, "nvfp4", "e2m1", "srelu", False), "tensor"),
    ("skewed", lambda: _meta("skewed", W.dirichlet_sizes(65536, 128, 0.1, seed=4), 7168, 4096, "mxfp8_e4m3",
                             "e4m3", "srelu", True), "tensor"),
    ("skinny", lambda: _meta("skinny", [t.size for t in W.route_softmax_topk(128, 64, 8, seed=7)[0]], 7168, 2048,
                             "mxfp8_e4m3", "bf16", "gate", False), "hbm"),
])
def test_workload_bounds(name, meta, bound):
    assert _bound(meta()) == bound


def test_skinny_routing():
    tokens, probs = W.route_softmax_topk(128, 64, 8, seed=7)
    counts = np.array([t.size for t in tokens])
    assert counts.sum() == 128 * 8
    assert counts.max() < 128                   # every group fits one 128-row tile
    p = _meta("skinny", counts, 7168, 2048, "mxfp8_e4m3", "bf16", "gate", False)
    nonempty = int((counts > 0).sum())
    assert p.m_pad == 128 * nonempty
    # the expert weights are almost all of the algorithmic bytes
    b_bytes = nonempty * 2048 * 7168
    assert b_bytes / bench.algorithmic_bytes(p) > 0.85
