"""Shared test helpers: hand problems to the oracle, and an independent
brute-force dequantizer (torch float8 decoding + the E2M1 listed values) used
to pin the oracle's GEMM."""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from block_scaled_grouped_gb300 import workloads as W

IN_CODE = {"mxfp8_e4m3": orc.IN_MXFP8_E4M3, "mxfp8_e5m2": orc.IN_MXFP8_E5M2, "nvfp4": orc.IN_NVFP4,
           "fp4_ue8m0_16": orc.IN_FP4_UE8M0_16, "mxfp4": orc.IN_MXFP4, "bf16": orc.IN_BF16}
OUT_CODE = {"bf16": orc.OUT_BF16, "f16": orc.OUT_F16, "f32": orc.OUT_F32, "e4m3": orc.OUT_E4M3,
            "e5m2": orc.OUT_E5M2, "e2m1": orc.OUT_E2M1}
EPI_CODE = {"gate": orc.EPI_GATE, "swiglu": orc.EPI_SWIGLU, "srelu": orc.EPI_SRELU, "geglu": orc.EPI_GEGLU,
            "dswiglu": orc.EPI_DSWIGLU, "dgeglu": orc.EPI_DGEGLU, "dsituglu": orc.EPI_DSITUGLU}

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def oracle_inputs(p: W.Problem) -> dict:
    return dict(
        a=np_(p.a), b=np_(p.b),
        sfa=orc.pack_sf(np_(p.sfa_rows)), sfb=orc.pack_sf(np_(p.sfb_rows)),
        padded_offsets=np_(p.padded_offsets), alpha=np_(p.alpha), prob=np_(p.prob))


def oracle_run(p: W.Problem, blocks=None, inputs=None, gate_first=0, threads=None, **over):
    ins = inputs if inputs is not None else oracle_inputs(p)
    ins = dict(ins)
    if p.epi in W.BWD_EPILOGUES:
        ins.setdefault("saved_c", np_(p.saved_c.double()))
        ins.setdefault("beta", np_(p.beta))
    ins.update(over)
    return orc.run(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups,
                   in_fmt=IN_CODE[p.in_fmt], out_fmt=OUT_CODE[p.out_fmt], epi=EPI_CODE[p.epi],
                   norm_const=p.norm_const, tanh_clamp_s=p.tanh_clamp_s, gate_first=gate_first,
                   want_col=p.want_col, blocks=blocks, threads=threads, **ins)


def dequant_dense(codes: np.ndarray, sf_rows: np.ndarray, in_fmt: str, k: int) -> np.ndarray:
    """Brute-force dequantization of a K-major operand with row-major scale
    codes (R, k/v), independent of the oracle's tables."""
    codes = np.ascontiguousarray(codes)
    if in_fmt == "bf16":
        # torch's bfloat16 decoding of the little-endian byte pairs; no scales
        return torch.from_numpy(codes).view(torch.bfloat16).double().numpy()[:, :k]
    if in_fmt in ("nvfp4", "fp4_ue8m0_16", "mxfp4"):
        lo = codes & 0xF
        hi = codes >> 4
        nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)[:, :k]
        vals = E2M1_VALUES[nib]
        sdt = torch.float8_e4m3fn if in_fmt == "nvfp4" else torch.float8_e8m0fnu
        sc = torch.from_numpy(np.ascontiguousarray(sf_rows)).view(sdt).double().numpy()
        v = 32 if in_fmt == "mxfp4" else 16
    else:
        dt = torch.float8_e4m3fn if in_fmt == "mxfp8_e4m3" else torch.float8_e5m2
        vals = torch.from_numpy(codes).view(dt).double().numpy()[:, :k]
        sc = torch.from_numpy(np.ascontiguousarray(sf_rows)).view(torch.float8_e8m0fnu).double().numpy()
        v = 32
    scale = np.repeat(sc, v, axis=1)[:, :k]
    return vals * scale


def brute_force_C(p: W.Problem) -> np.ndarray:
    """C = alpha_g * deq(A) @ deq(B_g)^T per group, rows outside groups = nan."""
    A = dequant_dense(np_(p.a), np_(p.sfa_rows)[0], p.in_fmt, p.k)
    off = np_(p.padded_offsets)
    alpha = np_(p.alpha)
    C = np.full((p.m_pad, p.n), np.nan)
    start = 0
    for g in range(p.num_groups):
        end = int(off[g])
        if end > start:
            Bg = dequant_dense(np_(p.b)[g], np_(p.sfb_rows)[g], p.in_fmt, p.k)
            C[start:end] = float(alpha[g]) * (A[start:end] @ Bg.T)
        start = end
    return C


def small_problem(counts=(70, 0, 130, 20), k=96, n=96, in_fmt="mxfp8_e4m3", out_fmt="bf16",
                  epi="gate", seed=11, pad_to=32, **kw) -> W.Problem:
    return W.build_problem(name="small", counts=list(counts), k=k, n=n, in_fmt=in_fmt,
                           out_fmt=out_fmt, epi=epi, seed=seed, pad_to=pad_to, **kw)
