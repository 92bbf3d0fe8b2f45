"""CPU parity oracle for the grouped block-scaled GEMM (test infrastructure).

The oracle is a plain, slow C++ implementation (``bsgg_oracle.cpp``): decode by
table, fp64 accumulation, the epilogue of the cuDNN-frontend pages in fp64 and
the output-quantization decisions in fp32.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the product library never does, and the two share no code.

This module only builds the shared object with g++ and marshals numpy arrays
through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsgg_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Format codes of the oracle (its own numbering, see bsgg_oracle.cpp).
F_E4M3, F_E5M2, F_E2M1, F_UE8M0 = 0, 1, 2, 3
IN_MXFP8_E4M3, IN_MXFP8_E5M2, IN_NVFP4, IN_FP4_UE8M0_16, IN_MXFP4, IN_BF16 = 0, 1, 2, 3, 4, 5
OUT_BF16, OUT_F16, OUT_F32, OUT_E4M3, OUT_E5M2, OUT_E2M1 = 0, 1, 2, 3, 4, 5
EPI_GATE, EPI_SWIGLU, EPI_SRELU, EPI_GEGLU, EPI_DSWIGLU, EPI_DGEGLU, EPI_DSITUGLU = 0, 1, 2, 3, 4, 5, 6
BWD_EPIS = (EPI_DSWIGLU, EPI_DGEGLU, EPI_DSITUGLU)


class OrcDesc(ctypes.Structure):
    _fields_ = [
        ("m_pad", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
        ("num_groups", ctypes.c_int64),
        ("in_fmt", ctypes.c_int32), ("out_fmt", ctypes.c_int32), ("epi", ctypes.c_int32),
        ("gate_first", ctypes.c_int32), ("want_col", ctypes.c_int32), ("rht", ctypes.c_int32),
        ("tanh_clamp_s", ctypes.c_double), ("glu_limit", ctypes.c_double), ("glu_alpha", ctypes.c_double),
        ("rht_norm", ctypes.c_double), ("geglu_alpha", ctypes.c_double), ("glu_clamp_min", ctypes.c_double),
        ("glu_clamp_max", ctypes.c_double), ("linear_offset", ctypes.c_double),
        ("situ_beta1", ctypes.c_double), ("situ_beta2", ctypes.c_double),
    ]


def compile_source(src: str, out: str) -> None:
    """Compile one copy of the oracle's source into a shared object with g++
    (plain C++17, no intrinsics, no fast-math)."""
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", out, src]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Compile the oracle (``oracle/_build/liboracle.so``) unless it is current."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def source_path() -> str:
    return _SRC


def lib():
    global _lib
    if _lib is None:
        # BSGG_ORACLE_LIB loads another build of this source instead: the
        # mutation test of the pins runs them against copies that each carry
        # one planted mistake.
        path = os.environ.get("BSGG_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        L.orc_decode.restype = ctypes.c_double
        L.orc_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
        L.orc_encode_rne_satfinite.restype = ctypes.c_uint32
        L.orc_encode_rne_satfinite.argtypes = [ctypes.c_int, ctypes.c_float]
        L.orc_encode_ue8m0_ceil.restype = ctypes.c_uint32
        L.orc_encode_ue8m0_ceil.argtypes = [ctypes.c_float]
        L.orc_sf_offset.restype = ctypes.c_int64
        L.orc_sf_offset.argtypes = [ctypes.c_int64] * 5
        L.orc_sf_bytes.restype = ctypes.c_int64
        L.orc_sf_bytes.argtypes = [ctypes.c_int64] * 3
        L.orc_pack_sf.restype = None
        L.orc_pack_sf.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_int64]
        L.orc_sigmoid.restype = ctypes.c_double
        L.orc_sigmoid.argtypes = [ctypes.c_double]
        L.orc_srelu.restype = ctypes.c_double
        L.orc_srelu.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_group_of_row.restype = ctypes.c_int64
        L.orc_group_of_row.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
        L.orc_run.restype = ctypes.c_int
        L.orc_run.argtypes = [ctypes.POINTER(OrcDesc)] + [ctypes.c_void_p] * 10 + [
            ctypes.c_float, ctypes.c_void_p, ctypes.c_int64] + [ctypes.c_void_p] * 12 + [ctypes.c_int]
        L.orc_round_bf16.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_hadamard16.restype = ctypes.c_double
        L.orc_hadamard16.argtypes = [ctypes.c_int, ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous numpy array"
    return a.ctypes.data


def decode(fmt: int, code: int) -> float:
    return lib().orc_decode(fmt, code)


def encode_rne_satfinite(fmt: int, x: float) -> int:
    return lib().orc_encode_rne_satfinite(fmt, x)


def encode_ue8m0_ceil(sf: float) -> int:
    return lib().orc_encode_ue8m0_ceil(sf)


def sf_offset(row: int, kblk: int, l: int, rows: int, kblocks: int) -> int:
    return lib().orc_sf_offset(row, kblk, l, rows, kblocks)


def sf_bytes(rows: int, kblocks: int, L: int) -> int:
    return lib().orc_sf_bytes(rows, kblocks, L)


def pack_sf(logical: np.ndarray) -> np.ndarray:
    """(L, rows, kblocks) uint8 -> flat swizzled uint8 buffer."""
    logical = np.ascontiguousarray(logical, dtype=np.uint8)
    L_, rows, kb = logical.shape
    out = np.empty(sf_bytes(rows, kb, L_), dtype=np.uint8)
    lib().orc_pack_sf(_ptr(logical), _ptr(out), rows, kb, L_)
    return out


def sigmoid(x: float) -> float:
    return lib().orc_sigmoid(x)


def srelu(c: float, s: float = 0.0) -> float:
    return lib().orc_srelu(c, s)


def group_of_row(offsets: np.ndarray, m: int) -> int:
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    return lib().orc_group_of_row(_ptr(off), off.size, m)


def round_bf16(x: float) -> float:
    return float(lib().orc_round_bf16(float(x)))


def hadamard16(i: int, j: int) -> float:
    return float(lib().orc_hadamard16(int(i), int(j)))


def n_out(n: int, epi: int) -> int:
    if epi in (EPI_SWIGLU, EPI_GEGLU):
        return n // 2
    return 2 * n if epi in BWD_EPIS else n


def run(*, m_pad, n, k, num_groups, in_fmt, out_fmt, epi, a, sfa, b, sfb, padded_offsets,
        alpha, prob, norm_const=1.0, tanh_clamp_s=0.0, gate_first=0, want_col=False,
        blocks=None, threads=None, outputs=None, bias=None, glu_limit=0.0, glu_alpha=1.0,
        want_c=False, saved_c=None, beta=None, rht=None, rht_norm=1.0, geglu_alpha=1.702,
        glu_clamp_min=-7.0, glu_clamp_max=7.0, linear_offset=1.0, situ_beta1=1.0, situ_beta2=1.0):
    """Run the oracle on the listed 32-row blocks (default: all of them).

    Inputs are numpy arrays in the device layouts: ``a`` (m_pad, k or k/2)
    uint8 codes (``IN_BF16``: (m_pad, 2k) bytes of little-endian bfloat16
    values, and no scales: ``sfa``/``sfb`` may be empty), ``b`` (L, n, k or
    k/2, or 2k), ``sfa``/``sfb`` swizzled flat uint8,
    ``padded_offsets`` int32 (L,), ``alpha`` float32 (L,), ``prob`` float32
    (m_pad,).  Returns a dict with ``d_ref`` (fp64, rows of the listed blocks),
    ``amax`` and, for quantized outputs, full-size ``d``, ``d_col``,
    ``sfd_row``, ``sfd_col`` buffers written for the listed rows only.
    ``bias`` (L, n) float32 is added to C; ``want_c`` adds ``c_ref`` (fp64 C of
    the listed rows, before any clamp or activation).  ``glu_limit`` (0 = none)
    and ``glu_alpha`` apply to SwiGLU and GeGLU.  The dSwiGLU backward
    (``epi=EPI_DSWIGLU``) takes ``saved_c`` (m_pad, 2n) values of the saved
    forward C (any float dtype, widened to fp64) and ``beta`` float32 (L,), and
    adds ``dprob_ref`` (fp64, rows of the listed blocks); its ``amax`` has 2L
    entries (input-gradient and gate-gradient blocks of each group).  The dGeGLU
    backward (``epi=EPI_DGEGLU``) takes the saved C unscaled (scaled by
    ``beta`` with ``IN_BF16``: the BF16 contract's X = beta C) and
    ``geglu_alpha``, ``glu_clamp_min``/``glu_clamp_max`` and ``linear_offset``
    (the page's defaults 1.702, -7, 7, 1); the dSiTU-GLU backward
    (``epi=EPI_DSITUGLU``) takes the saved C unscaled and ``situ_beta1``,
    ``situ_beta2``.  Every backward also returns ``dbias`` (L, 2n) fp64: the
    sum of D over the listed rows of each group.
    ``rht`` ("bf16" or "e2m1") adds the rowwise Hadamard output: ``rht_ref``
    (fp64) and, for "e2m1", full-size ``rht_q`` / ``sfrht`` buffers (E4M3
    scales per 16 under ``rht_norm``); "col_e2m1" the colwise one (16-token
    blocks per column, flat per-expert transposed ``rht_q`` and ``sfrht``).
    """
    L = lib()
    rht_code = {None: 0, "bf16": 1, "e2m1": 2, "col_e2m1": 3}[rht]
    desc = OrcDesc(m_pad, n, k, num_groups, in_fmt, out_fmt, epi, int(gate_first),
                   int(bool(want_col)), rht_code, float(tanh_clamp_s), float(glu_limit), float(glu_alpha),
                   float(rht_norm), float(geglu_alpha), float(glu_clamp_min), float(glu_clamp_max),
                   float(linear_offset), float(situ_beta1), float(situ_beta2))
    nd = n_out(n, epi)
    if blocks is None:
        blocks = np.arange(m_pad // 32, dtype=np.int64)
    blocks = np.ascontiguousarray(blocks, dtype=np.int64)
    if threads is None:
        threads = os.cpu_count() or 1
    d_ref = np.zeros((blocks.size * 32, nd), dtype=np.float64)
    c_ref = np.zeros((blocks.size * 32, n), dtype=np.float64) if want_c else None
    bias_arr = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(num_groups, n)
    bwd = epi in BWD_EPIS
    amax = np.zeros(2 * num_groups if bwd else num_groups, dtype=np.float32)
    rht_ref = np.zeros((blocks.size * 32, nd), dtype=np.float64) if rht_code else None
    dprob_ref = np.zeros(blocks.size * 32, dtype=np.float64) if bwd else None
    dbias = np.zeros((num_groups, nd), dtype=np.float64) if bwd else None
    saved_arr = None if saved_c is None else np.ascontiguousarray(saved_c, dtype=np.float64).reshape(m_pad, 2 * n)
    beta_arr = None if beta is None else np.ascontiguousarray(beta, dtype=np.float32).reshape(num_groups)
    outs = dict(outputs or {})
    if rht_code == 2:
        outs.setdefault("rht_q", np.zeros((m_pad, nd // 2), dtype=np.uint8))
        outs.setdefault("sfrht", np.zeros(sf_bytes(m_pad, -(-nd // 16), 1), dtype=np.uint8))
    if rht_code == 3:   # flat per-expert segments: m_pad * nd / 2 data bytes, m_pad * nd / 16 scales
        outs.setdefault("rht_q", np.zeros(m_pad * nd // 2, dtype=np.uint8))
        outs.setdefault("sfrht", np.zeros(m_pad * nd // 16, dtype=np.uint8))
    quant = out_fmt >= OUT_E4M3
    v = 16 if in_fmt in (IN_NVFP4, IN_FP4_UE8M0_16) else 32
    if quant:
        row_bytes = nd // 2 if out_fmt == OUT_E2M1 else nd
        outs.setdefault("d", np.zeros((m_pad, row_bytes), dtype=np.uint8))
        outs.setdefault("sfd_row", np.zeros(sf_bytes(m_pad, -(-nd // v), 1), dtype=np.uint8))
        if want_col:
            outs.setdefault("d_col", np.zeros((m_pad, row_bytes), dtype=np.uint8))
            outs.setdefault("sfd_col", np.zeros(sf_bytes(nd, -(-m_pad // v), 1), dtype=np.uint8))
    arrs = dict(
        a=np.ascontiguousarray(a, dtype=np.uint8), sfa=np.ascontiguousarray(sfa, dtype=np.uint8),
        b=np.ascontiguousarray(b, dtype=np.uint8), sfb=np.ascontiguousarray(sfb, dtype=np.uint8),
        off=np.ascontiguousarray(padded_offsets, dtype=np.int32),
        alpha=np.ascontiguousarray(alpha, dtype=np.float32),
        prob=np.ascontiguousarray(prob, dtype=np.float32).reshape(-1),
    )
    rc = L.orc_run(ctypes.byref(desc), _ptr(arrs["a"]), _ptr(arrs["sfa"]), _ptr(arrs["b"]),
                   _ptr(arrs["sfb"]), _ptr(arrs["off"]), _ptr(arrs["alpha"]), _ptr(arrs["prob"]),
                   _ptr(bias_arr), _ptr(saved_arr), _ptr(beta_arr), float(norm_const), _ptr(blocks),
                   blocks.size, _ptr(d_ref), _ptr(c_ref), _ptr(dprob_ref), _ptr(outs.get("d")),
                   _ptr(outs.get("d_col")), _ptr(outs.get("sfd_row")), _ptr(outs.get("sfd_col")),
                   _ptr(amax), _ptr(rht_ref), _ptr(outs.get("rht_q")), _ptr(outs.get("sfrht")), _ptr(dbias),
                   int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    res = {"d_ref": d_ref, "amax": amax, "blocks": blocks}
    if want_c:
        res["c_ref"] = c_ref
    if dprob_ref is not None:
        res["dprob_ref"] = dprob_ref
        res["dbias"] = dbias
    if rht_ref is not None:
        res["rht_ref"] = rht_ref
    res.update(outs)
    return res
