"""GB300 grouped block-scaled GEMM with fused MoE epilogue (Python binding).

A thin ctypes binding over the C ABI in ``include/bsgg.h`` (library
``_build/libbsgg.so``, built by ``build.py``).  It only marshals arguments:
device pointers are taken from torch tensors, streams from torch's current
stream.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU path, and calls fail loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

IN_FORMATS = {"mxfp8_e4m3": 0, "mxfp8_e5m2": 1, "nvfp4": 2, "fp4_ue8m0_16": 3, "mxfp4": 4, "bf16": 5}
OUT_FORMATS = {"bf16": 0, "f16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "e2m1": 5}
EPILOGUES = {"gate": 0, "swiglu": 1, "srelu": 2, "geglu": 3, "dswiglu": 4, "dgeglu": 5, "dsituglu": 6}
BWD_EPILOGUES = ("dswiglu", "dgeglu", "dsituglu")
GLU_EPILOGUES = ("swiglu", "geglu")
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
          4: "device wait timed out", 5: "padded_offsets invalid", 6: "expert weight pointer invalid",
          7: "an index failed its range check"}

SYMBOLS = ("bsgg_create", "bsgg_run", "bsgg_run_host", "bsgg_run_host_async", "bsgg_query_device_status",
           "bsgg_destroy",
           "bsgg_status_string", "bsgg_sf_bytes", "bsgg_sf_offset", "bsgg_pack_sf", "bsgg_run_noalloc",
           "bsgg_measure_mma_peak", "bsgg_measure_mma_peak_tile", "bsgg_debug_force_timeout",
           "bsgg_launches_per_run", "bsgg_debug_bounds_checked", "bsgg_debug_bounds_margin",
           "bsgg_debug_bounds_violation")


class BsggError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class Desc(ctypes.Structure):
    _fields_ = [("m_pad", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("num_groups", ctypes.c_int32), ("in_format", ctypes.c_int32),
                ("out_format", ctypes.c_int32), ("epilogue", ctypes.c_int32),
                ("want_col", ctypes.c_int32), ("gate_first", ctypes.c_int32),
                ("tanh_clamp_s", ctypes.c_float), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("cluster_m", ctypes.c_int32), ("cluster_n", ctypes.c_int32),
                ("glu_limit", ctypes.c_float), ("glu_alpha", ctypes.c_float),
                ("want_c", ctypes.c_int32), ("c_format", ctypes.c_int32),
                ("want_bias", ctypes.c_int32), ("bias_format", ctypes.c_int32),
                ("discrete_b", ctypes.c_int32), ("saved_c_format", ctypes.c_int32),
                ("want_rht", ctypes.c_int32), ("rht_format", ctypes.c_int32),
                ("dgeglu_custom", ctypes.c_int32), ("dgeglu_alpha", ctypes.c_float),
                ("dgeglu_clamp_min", ctypes.c_float), ("dgeglu_clamp_max", ctypes.c_float),
                ("dgeglu_linear_offset", ctypes.c_float), ("situ_beta1", ctypes.c_float),
                ("situ_beta2", ctypes.c_float)]


def make_desc(*, m_pad: int, n: int, k: int, num_groups: int, in_format: str, out_format: str,
              epilogue: str, want_col: bool = False, gate_first: bool = False,
              tanh_clamp_s: float = 0.0, tile=(0, 0), cluster=(0, 0), glu_limit: float = 0.0,
              glu_alpha: float = 0.0, c_format: Optional[str] = None,
              bias_format: Optional[str] = None, discrete_b: bool = False,
              saved_c_format: str = "bf16", rht_format: Optional[str] = None,
              dgeglu_params: Optional[tuple] = None, situ_betas: Optional[tuple] = None,
              rht_colwise: bool = False) -> "Desc":
    """A bsgg_desc.  c_format ("bf16"/"f16"; with MXFP8 inputs also "f32",
    "e4m3", "e5m2", "e2m1") asks for the pre-activation C
    output, bias_format ("bf16"/"f16"/"f32") for a bias; None = neither.
    discrete_b: per-expert weights through the b_ptrs / sfb_ptrs arrays.
    saved_c_format: storage type of the saved C read by the dSwiGLU backward.
    rht_format ("bf16"/"e2m1"): the rowwise Hadamard output; None = none;
    with rht_colwise the colwise one (e2m1, per-expert transposed).
    dgeglu_params: (geglu_alpha, clamp_min, clamp_max, linear_offset) of the
    dGeGLU backward; None = the page's defaults (1.702, -7, 7, 1).
    situ_betas: (beta1, beta2) of the dSiTU-GLU backward; None = (1, 1)."""
    dg = tuple(float(x) for x in dgeglu_params) if dgeglu_params is not None else (0.0, 0.0, 0.0, 0.0)
    return Desc(m_pad, n, k, num_groups, IN_FORMATS[in_format], OUT_FORMATS[out_format],
                EPILOGUES[epilogue], int(bool(want_col)), int(bool(gate_first)), float(tanh_clamp_s),
                int(tile[0]), int(tile[1]), int(cluster[0]), int(cluster[1]), float(glu_limit),
                float(glu_alpha), int(c_format is not None), OUT_FORMATS[c_format or "bf16"],
                int(bias_format is not None), OUT_FORMATS[bias_format or "bf16"], int(bool(discrete_b)),
                OUT_FORMATS[saved_c_format], (2 if rht_colwise else 1) if rht_format is not None else 0,
                OUT_FORMATS[rht_format or "bf16"],
                int(dgeglu_params is not None), *dg,
                *(tuple(float(x) for x in situ_betas) if situ_betas is not None else (0.0, 0.0)))


class Args(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "a", "sfa", "b", "sfb", "padded_offsets", "alpha", "prob", "norm_const",
        "d", "d_col", "sfd_row", "sfd_col", "amax", "bias", "c", "b_ptrs", "sfb_ptrs", "saved_c", "beta",
        "dprob", "rht", "sfrht", "rht_norm_const", "dbias")]


_libs = {}


def library_path(debug_bounds: bool = False) -> str:
    return _build.DEBUG_LIB_PATH if debug_bounds else _build.LIB_PATH


def lib(debug_bounds: bool = False):
    """Load libbsgg.so, or with debug_bounds the range-checking build
    libbsgg_debug.so (raises if it has not been built)."""
    L = _libs.get(debug_bounds)
    if L is None:
        path = library_path(debug_bounds)
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run block_scaled_grouped_gb300.build")
        L = ctypes.CDLL(path)
        L.bsgg_create.restype = ctypes.c_int
        L.bsgg_create.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(ctypes.c_void_p)]
        L.bsgg_run.restype = ctypes.c_int
        L.bsgg_run.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.c_void_p]
        L.bsgg_run_host.restype = ctypes.c_int
        L.bsgg_run_host.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.POINTER(Args),
                                    ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64),
                                    ctypes.POINTER(ctypes.c_uint64)]
        L.bsgg_run_host_async.restype = ctypes.c_int
        L.bsgg_run_host_async.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.POINTER(Args),
                                          ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64),
                                          ctypes.POINTER(ctypes.c_uint64)]
        L.bsgg_query_device_status.restype = ctypes.c_int
        L.bsgg_query_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        L.bsgg_destroy.restype = None
        L.bsgg_destroy.argtypes = [ctypes.c_void_p]
        L.bsgg_status_string.restype = ctypes.c_char_p
        L.bsgg_status_string.argtypes = [ctypes.c_int]
        L.bsgg_sf_bytes.restype = ctypes.c_uint64
        L.bsgg_sf_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        L.bsgg_sf_offset.restype = ctypes.c_int64
        L.bsgg_sf_offset.argtypes = [ctypes.c_int64] * 5
        L.bsgg_run_noalloc.restype = ctypes.c_int
        L.bsgg_run_noalloc.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Args), ctypes.c_void_p,
                                       ctypes.c_int32]
        L.bsgg_measure_mma_peak.restype = ctypes.c_int
        L.bsgg_measure_mma_peak.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                            ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
        L.bsgg_measure_mma_peak_tile.restype = ctypes.c_int
        L.bsgg_measure_mma_peak_tile.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
        L.bsgg_debug_force_timeout.restype = ctypes.c_int
        L.bsgg_debug_force_timeout.argtypes = [ctypes.c_void_p, ctypes.c_int32]
        L.bsgg_launches_per_run.restype = ctypes.c_int32
        L.bsgg_launches_per_run.argtypes = [ctypes.c_void_p]
        L.bsgg_pack_sf.restype = ctypes.c_int
        L.bsgg_pack_sf.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int32, ctypes.c_void_p]
        L.bsgg_debug_bounds_checked.restype = ctypes.c_int32
        L.bsgg_debug_bounds_checked.argtypes = []
        L.bsgg_debug_bounds_margin.restype = ctypes.c_int
        L.bsgg_debug_bounds_margin.argtypes = [ctypes.c_void_p, ctypes.c_int32]
        L.bsgg_debug_bounds_violation.restype = ctypes.c_int
        L.bsgg_debug_bounds_violation.argtypes = [ctypes.c_void_p] + [ctypes.POINTER(ctypes.c_uint32)] * 3
        _libs[debug_bounds] = L
    return L


def _check(code: int, what: str) -> None:
    if code != 0:
        raise BsggError(code, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def sf_bytes(rows: int, cols: int, sf_vec: int, num_slices: int = 1) -> int:
    return int(lib().bsgg_sf_bytes(rows, cols, sf_vec, num_slices))


def sf_offset(row: int, kblk: int, l: int, rows: int, kblocks: int) -> int:
    return int(lib().bsgg_sf_offset(row, kblk, l, rows, kblocks))


def pack_sf(rowmajor, out=None, stream=None):
    """Pack (L, rows, kblocks) uint8 scale codes (device tensor) into the
    swizzled layout (flat uint8 device tensor)."""
    import torch
    L_, rows, kb = rowmajor.shape
    assert rowmajor.is_cuda and rowmajor.dtype == torch.uint8 and rowmajor.is_contiguous()
    if kb == 0:   # no scale factors (bf16 operands): nothing to pack
        return torch.empty(0, dtype=torch.uint8, device=rowmajor.device)
    nbytes = sf_bytes(rows, kb, 1, L_)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=rowmajor.device)
    assert out.numel() >= nbytes
    _check(lib().bsgg_pack_sf(_ptr(rowmajor), _ptr(out), rows, kb, L_, _stream(stream)), "bsgg_pack_sf")
    return out


class Plan:
    """A validated problem description (bsgg_create); run() launches it."""

    def __init__(self, debug_bounds: bool = False, **kw):
        """Keyword arguments of make_desc.  tile = the pages' mma_tiler_mn,
        cluster = cluster_shape_mn; (0, 0) lets the library choose.
        debug_bounds: create and run the plan in the range-checking build
        (libbsgg_debug.so)."""
        self._lib = lib(debug_bounds)
        self.desc = make_desc(**kw)
        self.in_format, self.out_format, self.epilogue = kw["in_format"], kw["out_format"], kw["epilogue"]
        self.want_col = bool(kw.get("want_col", False))
        self.c_format = kw.get("c_format")
        self.rht_format = kw.get("rht_format")
        self.rht_colwise = bool(kw.get("rht_colwise", False))
        h = ctypes.c_void_p()
        _check(self._lib.bsgg_create(ctypes.byref(self.desc), ctypes.byref(h)), "bsgg_create")
        self._h = h

    # shapes --------------------------------------------------------------
    @property
    def sf_vec(self) -> int:
        return 16 if self.in_format in ("nvfp4", "fp4_ue8m0_16") else 32

    @property
    def n_out(self) -> int:
        if self.epilogue in GLU_EPILOGUES:
            return self.desc.n // 2
        return 2 * self.desc.n if self.epilogue in BWD_EPILOGUES else self.desc.n

    @property
    def out_row_bytes(self) -> int:
        bits = {"bf16": 16, "f16": 16, "f32": 32, "e4m3": 8, "e5m2": 8, "e2m1": 4}[self.out_format]
        return self.n_out * bits // 8

    @property
    def quantized(self) -> bool:
        return self.out_format in ("e4m3", "e5m2", "e2m1")

    def output_bytes(self) -> dict:
        d = self.desc
        out = {"d": d.m_pad * self.out_row_bytes}
        if self.quantized:
            out["sfd_row"] = sf_bytes(d.m_pad, self.n_out, self.sf_vec, 1)
            if self.want_col:
                out["d_col"] = out["d"]
                out["sfd_col"] = sf_bytes(self.n_out, d.m_pad, self.sf_vec, 1)
        else:
            out["amax"] = 4 * d.num_groups * (2 if self.epilogue in BWD_EPILOGUES else 1)
        if self.c_format is not None:
            bits = {"bf16": 16, "f16": 16, "f32": 32, "e4m3": 8, "e5m2": 8, "e2m1": 4}[self.c_format]
            out["c"] = d.m_pad * d.n * bits // 8
        if self.rht_format == "bf16":
            out["rht"] = d.m_pad * self.n_out * 2
        elif self.rht_format == "e2m1":
            out["rht"] = d.m_pad * self.n_out // 2
            out["sfrht"] = (d.m_pad * self.n_out // 16 if self.rht_colwise
                            else sf_bytes(d.m_pad, self.n_out, 16, 1))
        return out

    # calls ---------------------------------------------------------------
    def _args(self, t: dict) -> Args:
        return Args(*[_ptr(t.get(name)) for name, _ in Args._fields_])

    def run(self, stream=None, **tensors) -> None:
        """Enqueue the kernel; tensors by the bsgg_args names (device)."""
        args = self._args(tensors)
        _check(self._lib.bsgg_run(self._h, ctypes.byref(args), _stream(stream)), "bsgg_run")

    def run_host(self, host: dict, dev: dict, stream=None, sync: bool = True):
        """Host-buffer call: copies host inputs in, runs, copies outputs out
        and, with sync, synchronizes (bsgg_run_host; without sync
        bsgg_run_host_async, whose outputs are complete once `stream` has
        finished).  Returns (h2d_bytes, d2h_bytes)."""
        hi, di = self._args(host), self._args(dev)
        h2d, d2h = ctypes.c_uint64(), ctypes.c_uint64()
        fn = self._lib.bsgg_run_host if sync else self._lib.bsgg_run_host_async
        _check(fn(self._h, ctypes.byref(hi), ctypes.byref(di), _stream(stream), ctypes.byref(h2d),
                  ctypes.byref(d2h)), "bsgg_run_host" if sync else "bsgg_run_host_async")
        return int(h2d.value), int(d2h.value)

    @property
    def launches_per_run(self) -> int:
        """Kernel launches one run() enqueues (bsgg_launches_per_run)."""
        return int(self._lib.bsgg_launches_per_run(self._h))

    def device_status(self, stream=None) -> int:
        """Synchronize and read/clear the device status word (0 = ok)."""
        return int(self._lib.bsgg_query_device_status(self._h, _stream(stream)))

    def debug_force_timeout(self, enable: bool) -> None:
        """Test hook (bsgg_debug_force_timeout): later launches give up after a
        forced barrier timeout and report BSGG_ERR_DEVICE_TIMEOUT."""
        _check(self._lib.bsgg_debug_force_timeout(self._h, int(bool(enable))), "bsgg_debug_force_timeout")

    def debug_bounds_margin(self, rows: int) -> None:
        """Test hook of the range-checking build (bsgg_debug_bounds_margin)."""
        _check(self._lib.bsgg_debug_bounds_margin(self._h, int(rows)), "bsgg_debug_bounds_margin")

    def debug_bounds_violation(self) -> tuple:
        """(site, value, limit) of the last range-check failure read back."""
        v = [ctypes.c_uint32() for _ in range(3)]
        _check(self._lib.bsgg_debug_bounds_violation(self._h, *[ctypes.byref(x) for x in v]),
               "bsgg_debug_bounds_violation")
        return tuple(int(x.value) for x in v)

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.bsgg_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def measure_mma_peak(in_format: str, tile_n: int = 256, mmas_per_sm: int = 400000, stream=None) -> float:
    """bsgg_measure_mma_peak: TFLOP/s of back-to-back block-scaled MMAs on
    resident operands (no loads, no epilogue) on the current device."""
    out = ctypes.c_double()
    _check(lib().bsgg_measure_mma_peak(IN_FORMATS[in_format], int(tile_n), int(mmas_per_sm),
                                       ctypes.byref(out), _stream(stream)), "bsgg_measure_mma_peak")
    return float(out.value)


def measure_mma_peak_tile(in_format: str, tile_m: int = 256, tile_n: int = 256, mmas: int = 400000,
                          stream=None) -> float:
    """bsgg_measure_mma_peak_tile: the same for the cta_group::1 (tile_m = 128)
    or cta_group::2 (tile_m = 256, tile_n = 256, an SM pair) instruction form."""
    out = ctypes.c_double()
    _check(lib().bsgg_measure_mma_peak_tile(IN_FORMATS[in_format], int(tile_m), int(tile_n), int(mmas),
                                            ctypes.byref(out), _stream(stream)), "bsgg_measure_mma_peak_tile")
    return float(out.value)


_DESC_KEYS = ("m_pad", "n", "k", "num_groups", "in_format", "out_format", "epilogue", "want_col",
              "gate_first", "tanh_clamp_s", "tile", "cluster", "glu_limit", "glu_alpha", "c_format",
              "bias_format", "discrete_b", "saved_c_format", "rht_format", "dgeglu_params", "situ_betas",
              "rht_colwise")


def run_noalloc(*, stream=None, wait_status: bool = True, **kw) -> int:
    """bsgg_run_noalloc: one call without a plan and without any device
    allocation (for callers whose device memory is owned by someone else, or
    who must not let cudaMalloc synchronize the device).  Keyword arguments:
    those of make_desc plus the tensors by their bsgg_args names.  Returns the
    status code (the device status when wait_status is true)."""
    desc = make_desc(**{k_: v for k_, v in kw.items() if k_ in _DESC_KEYS})
    tensors = {k_: v for k_, v in kw.items() if k_ not in _DESC_KEYS}
    args = Args(*[_ptr(tensors.get(name)) for name, _ in Args._fields_])
    return int(lib().bsgg_run_noalloc(ctypes.byref(desc), ctypes.byref(args), _stream(stream),
                                      int(bool(wait_status))))
