"""GPU-side helpers for the parity tests: run a workloads.Problem through the
C ABI (device buffers from torch) and compare the outputs with the oracle's."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_grouped_gb300 as bsgg
from block_scaled_grouped_gb300 import workloads as W

SENTINEL = 0x5A


def to_device(p: W.Problem, device="cuda") -> W.Problem:
    if p.a.is_cuda:
        return p
    import dataclasses
    return dataclasses.replace(
        p, padded_offsets=p.padded_offsets.to(device), alpha=p.alpha.to(device),
        prob=p.prob.to(device), a=p.a.to(device), sfa_rows=p.sfa_rows.to(device),
        b=p.b.to(device), sfb_rows=p.sfb_rows.to(device),
        saved_c=None if p.saved_c is None else p.saved_c.to(device),
        beta=None if p.beta is None else p.beta.to(device))


# (tile_m, tile_n, cluster_m, cluster_n): single CTA 128 x 128 and 128 x 256,
# and 256 x 256 CTA pairs
TILES = [(128, 128, 1, 1), (128, 256, 1, 1), (256, 256, 2, 1)]


def tile_id(t) -> str:
    if tuple(t[:2]) == (0, 0):
        return "default"
    return f"{t[0]}x{t[1]}" + (f"c{t[2]}x{t[3]}" if len(t) > 2 else "")


def make_plan(p: W.Problem, gate_first=False, tile=(0, 0)) -> bsgg.Plan:
    """tile: (tile_m, tile_n) or (tile_m, tile_n, cluster_m, cluster_n)."""
    cluster = tuple(tile[2:4]) if len(tile) > 2 else (0, 0)
    return bsgg.Plan(m_pad=p.m_pad, n=p.n, k=p.k, num_groups=p.num_groups, in_format=p.in_fmt,
                     out_format=p.out_fmt, epilogue=p.epi, want_col=p.want_col,
                     gate_first=gate_first, tanh_clamp_s=p.tanh_clamp_s, tile=tuple(tile[:2]),
                     cluster=cluster)


def alloc_outputs(plan: bsgg.Plan, device="cuda") -> dict:
    out = {}
    for name, nbytes in plan.output_bytes().items():
        if name == "amax":
            out[name] = torch.full((nbytes // 4,), -1.0, dtype=torch.float32, device=device)
        else:
            out[name] = torch.full((nbytes,), SENTINEL, dtype=torch.uint8, device=device)
    return out


def run_gpu(p: W.Problem, plan: bsgg.Plan = None, gate_first=False, outputs=None, inputs=None, tile=(0, 0)):
    """Pack the scales with the library's packer, launch, check the device
    status word.  Returns (outputs dict of device tensors, packed sfa, sfb)."""
    p = to_device(p)
    plan = plan or make_plan(p, gate_first, tile)
    if inputs is None:
        sfa = bsgg.pack_sf(p.sfa_rows)
        sfb = bsgg.pack_sf(p.sfb_rows)
    else:
        sfa, sfb = inputs
    outs = outputs if outputs is not None else alloc_outputs(plan)
    norm = torch.tensor([p.norm_const], dtype=torch.float32, device="cuda")
    plan.run(a=p.a, sfa=sfa, b=p.b, sfb=sfb, padded_offsets=p.padded_offsets, alpha=p.alpha,
             prob=p.prob, norm_const=norm, **outs)
    st = plan.device_status()
    assert st == 0, f"device status {st}"
    return outs, sfa, sfb


# --------------------------------------------------------------------------
# comparisons
# --------------------------------------------------------------------------

def decode_float_out(raw: np.ndarray, out_fmt: str, m_pad: int, n_out: int) -> np.ndarray:
    if out_fmt == "bf16":
        t = torch.from_numpy(raw.copy()).view(torch.bfloat16)
    elif out_fmt == "f16":
        t = torch.from_numpy(raw.copy()).view(torch.float16)
    else:
        t = torch.from_numpy(raw.copy()).view(torch.float32)
    return t.double().numpy().reshape(m_pad, n_out)


def check_float_d(d_gpu: np.ndarray, d_ref: np.ndarray, what="D"):
    """|d - ref| <= 2^-7 |ref| + 1e-3 rms(ref), element by element."""
    rms = float(np.sqrt(np.mean(d_ref ** 2))) if d_ref.size else 0.0
    tol = 2.0 ** -7 * np.abs(d_ref) + 1e-3 * rms
    err = np.abs(d_gpu - d_ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first "
                             f"{[(tuple(i), d_gpu[tuple(i)], d_ref[tuple(i)]) for i in idx]}")


def code_rank(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Order-preserving integer of a signed FP code (+0 and -0 both 0)."""
    codes = codes.astype(np.int64)
    if fmt == "e2m1":
        sign, mag = (codes >> 3) & 1, codes & 7
    else:
        sign, mag = (codes >> 7) & 1, codes & 0x7F
    return np.where(sign == 1, -mag, mag)


def unpack_e2m1(raw: np.ndarray, rows: int, n: int) -> np.ndarray:
    b = raw.reshape(rows, n // 2)
    return np.stack([b & 0xF, b >> 4], axis=-1).reshape(rows, n)


def check_codes(got: np.ndarray, ref: np.ndarray, fmt: str, what: str, min_equal=0.999):
    """>= 99.9% bit-equal, the rest within one code step."""
    if got.size == 0:
        return
    eq = got == ref
    frac = float(eq.mean())
    step = np.abs(code_rank(got, fmt) - code_rank(ref, fmt))
    assert frac >= min_equal, f"{what}: only {frac:.5f} of codes equal"
    assert int(step.max()) <= 1, f"{what}: a code is {int(step.max())} steps off"


def check_sf_codes(got: np.ndarray, ref: np.ndarray, what: str, min_equal=0.999):
    """Scale codes (UE8M0 or positive E4M3): >= 99.9% equal, the rest one step."""
    if got.size == 0:
        return
    eq = got == ref
    assert float(eq.mean()) >= min_equal, f"{what}: only {float(eq.mean()):.5f} equal"
    assert int(np.abs(got.astype(np.int64) - ref.astype(np.int64)).max()) <= 1, f"{what}: > 1 step"


def _sf_value(codes: np.ndarray, in_fmt: str) -> np.ndarray:
    dt = torch.float8_e4m3fn if in_fmt == "nvfp4" else torch.float8_e8m0fnu   # UE8M0 for MXFP8 and the UE8M0 FP4 forms
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(dt).double().numpy()


def _out_value(codes: np.ndarray, fmt: str) -> np.ndarray:
    from helpers import E2M1_VALUES
    if fmt == "e2m1":
        return E2M1_VALUES[codes]
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(dt).double().numpy()


MANT_BITS = {"e4m3": 3, "e5m2": 2, "e2m1": 1}


def _check_quant_plane(gq, rq, gsf, rsf, d_ref, fmt, in_fmt, norm, v, axis, what):
    """gq/rq: (rows, cols) codes; gsf/rsf: scale codes per block, shaped
    (rows, cols/v) for axis=1 (row blocks) or (rows/v, cols) for axis=0."""
    check_sf_codes(gsf, rsf, what + " scales")
    same = np.repeat(gsf == rsf, v, axis=axis)
    # blocks with equal scales: codes compared directly
    check_codes(gq[same], rq[same], fmt, what)
    # blocks whose scale is one step off: dequantized values within one
    # top-of-range output step of the block maximum
    if (~same).any():
        gval = _out_value(gq, fmt) * np.repeat(_sf_value(gsf, in_fmt), v, axis=axis) / norm
        rval = _out_value(rq, fmt) * np.repeat(_sf_value(rsf, in_fmt), v, axis=axis) / norm
        if axis == 1:
            am = np.abs(d_ref).reshape(d_ref.shape[0], -1, v).max(-1)
        else:
            am = np.abs(d_ref).reshape(-1, v, d_ref.shape[1]).max(1)
        amr = np.repeat(am, v, axis=axis)
        tol = 2.0 ** -MANT_BITS[fmt] * amr * 1.0001
        bad = (~same) & (np.abs(gval - rval) > tol)
        assert not bad.any(), f"{what}: {int(bad.sum())} values off in blocks with differing scales"


def compare(p: W.Problem, outs: dict, ref: dict, blocks=None):
    """Element-by-element parity of a GPU run against the oracle's result on
    the listed 32-row blocks (all blocks when None)."""
    import oracle as orc
    m_pad, nd = p.m_pad, p.n_out
    if blocks is None:
        blocks = np.arange(m_pad // 32)
    blocks = np.asarray(blocks)
    rows = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    off = p.padded_offsets.cpu().numpy()
    in_grp = rows < off[-1]
    rows, d_ref = rows[in_grp], ref["d_ref"][in_grp]
    if p.out_fmt in ("bf16", "f16", "f32"):
        raw = outs["d"].cpu().numpy()
        d = decode_float_out(raw, p.out_fmt, m_pad, nd)[rows]
        check_float_d(d, d_ref)
        return
    v = p.sf_vec
    g_d = outs["d"].cpu().numpy().reshape(m_pad, -1)
    r_d = ref["d"].reshape(m_pad, -1)
    if p.out_fmt == "e2m1":
        g_d, r_d = unpack_e2m1(g_d, m_pad, nd), unpack_e2m1(r_d, m_pad, nd)
    kb = nd // v
    offs = np.array([[orc.sf_offset(r, j, 0, m_pad, kb) for j in range(kb)] for r in rows])
    g_sf = outs["sfd_row"].cpu().numpy()[offs]
    r_sf = ref["sfd_row"][offs]
    _check_quant_plane(g_d[rows], r_d[rows], g_sf, r_sf, d_ref, p.out_fmt, p.in_fmt, p.norm_const,
                       v, 1, "D/SFD_row")
    if p.want_col:
        g_c = outs["d_col"].cpu().numpy().reshape(m_pad, -1)
        r_c = ref["d_col"].reshape(m_pad, -1)
        if p.out_fmt == "e2m1":
            g_c, r_c = unpack_e2m1(g_c, m_pad, nd), unpack_e2m1(r_c, m_pad, nd)
        # column blocks are whole 32-row blocks of the listed rows
        cb = np.unique(rows // v)
        kbc = -(-m_pad // v)
        offs_c = np.array([[orc.sf_offset(j, b, 0, nd, kbc) for j in range(nd)] for b in cb])
        g_sfc = outs["sfd_col"].cpu().numpy()[offs_c]
        r_sfc = ref["sfd_col"][offs_c]
        crow = (cb[:, None] * v + np.arange(v)[None, :]).reshape(-1)
        # d_ref rows in the order of crow
        pos = {int(r): i for i, r in enumerate(rows)}
        d_ref_c = d_ref[[pos[int(r)] for r in crow]]
        _check_quant_plane(g_c[crow], r_c[crow], g_sfc, r_sfc, d_ref_c, p.out_fmt, p.in_fmt,
                           p.norm_const, v, 0, "D_col/SFD_col")
