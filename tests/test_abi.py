"""The C ABI without a GPU: the library loads, exports every entry point
include/bsgg.h declares, its host-only helpers agree with the oracle's layout
map, and bsgg_create rejects what the pages' constraints reject (validation
runs before any device call)."""
import ctypes
import os
import re

import pytest

import block_scaled_grouped_gb300 as bsgg
from block_scaled_grouped_gb300 import build as bsgg_build
import oracle as orc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bsgg.h")


@pytest.fixture(scope="module")
def lib():
    bsgg_build.build()
    return bsgg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsgg_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(bsgg.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_range_checking_build_exports_the_same_symbols(lib):
    """libbsgg_debug.so (-DBSGG_DEBUG_BOUNDS) has the same entry points; only it
    reports the checks as compiled in, and only it accepts a test margin."""
    bsgg_build.build(debug_bounds=True)
    dbg = bsgg.lib(debug_bounds=True)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.bsgg_debug_bounds_checked() == 1
    assert lib.bsgg_debug_bounds_checked() == 0
    assert lib.bsgg_debug_bounds_margin(None, 0) == 1 and dbg.bsgg_debug_bounds_margin(None, 0) == 1
    assert lib.bsgg_debug_bounds_violation(None, None, None, None) == 1


def test_status_strings(lib):
    for code, text in bsgg.STATUS.items():
        assert lib.bsgg_status_string(code).decode() == text


def test_sf_helpers_match_the_oracle(lib):
    for rows, cols, v, L in [(384, 256, 32, 1), (4096, 7168, 16, 3), (100, 96, 32, 2)]:
        kb = -(-cols // v)
        assert bsgg.sf_bytes(rows, cols, v, L) == orc.sf_bytes(rows, kb, L)
        for (r, k, l) in [(0, 0, 0), (rows - 1, kb - 1, L - 1), (37, kb // 2, L // 2), (129, 5 % kb, 0)]:
            assert bsgg.sf_offset(r, k, l, rows, kb) == orc.sf_offset(r, k, l, rows, kb)


def _create(**over):
    """bsgg_create's status for the default description with `over` applied;
    a plan it makes is destroyed at once."""
    d = dict(m_pad=384, n=256, k=256, num_groups=2, in_format="mxfp8_e4m3", out_format="bf16",
             epilogue="gate")
    raw = {k_: over.pop(k_) for k_ in ("c_format_code", "bias_format_code", "want_c_raw", "discrete_raw")
           if k_ in over}
    d.update(over)
    tile = (d.pop("tile_m", 0), d.pop("tile_n", 0))
    cluster = (d.pop("cluster_m", 0), d.pop("cluster_n", 0))
    desc = bsgg.make_desc(tile=tile, cluster=cluster, **d)
    # raw enum values the Python names cannot express
    if "c_format_code" in raw:
        desc.want_c, desc.c_format = 1, raw["c_format_code"]
    if "bias_format_code" in raw:
        desc.want_bias, desc.bias_format = 1, raw["bias_format_code"]
    if "want_c_raw" in raw:
        desc.want_c = raw["want_c_raw"]
    if "discrete_raw" in raw:
        desc.discrete_b = raw["discrete_raw"]
    h = ctypes.c_void_p()
    code = bsgg.lib().bsgg_create(ctypes.byref(desc), ctypes.byref(h))
    if h.value:
        bsgg.lib().bsgg_destroy(h)
    return code


@pytest.mark.parametrize("over,code", [
    (dict(m_pad=200), 1),                       # groups are padded to 128 rows
    (dict(m_pad=0), 1),                         # an all-empty batch: refused, no zero-row descriptors
    (dict(m_pad=-128), 1),
    (dict(num_groups=0), 1), (dict(num_groups=1025), 1),   # L <= 1024
    (dict(k=40), 1),                            # 16-byte K-major rows
    (dict(k=48, in_format="nvfp4"), 1),         # FP4: K % 32
    (dict(n=96, epilogue="swiglu"), 1),         # SwiGLU pairs 32-column blocks: N % 64
    (dict(n=80), 1),                            # outputs in 32-column chunks
    (dict(tanh_clamp_s=-1.0, epilogue="srelu"), 1),
    (dict(tanh_clamp_s=8.0, epilogue="gate"), 1),
    (dict(want_col=1, out_format="bf16"), 1),   # D_col only with quantized outputs
    (dict(tile_m=64), 1), (dict(tile_n=192), 1),
    (dict(tile_m=256, tile_n=128), 2),           # pairs are built for 256 x 256 tiles
    (dict(cluster_m=1), 1), (dict(cluster_n=1), 1),          # cluster shape: both or neither
    (dict(cluster_m=3, cluster_n=1), 1), (dict(cluster_m=8, cluster_n=1), 1),   # powers of 2 <= 4
    (dict(tile_m=256, cluster_m=1, cluster_n=1), 1),         # 2-CTA tiles need an even CLUSTER_M
    (dict(cluster_m=4, cluster_n=1), 2), (dict(cluster_m=1, cluster_n=2), 2),   # valid, not built
    # (2, 1) clusters of 128-row or 128-column tiles would share an operand by
    # TMA multicast, which this library does not issue
    (dict(tile_m=128, tile_n=128, cluster_m=2, cluster_n=1), 2),
    (dict(tile_m=128, tile_n=256, cluster_m=2, cluster_n=1), 2),
    (dict(tile_m=128, tile_n=256, cluster_m=2, cluster_n=1, in_format="nvfp4"), 2),
    (dict(tile_m=128, tile_n=256, cluster_m=2, cluster_n=1, epilogue="dswiglu"), 2),
    (dict(tile_n=128, cluster_m=2, cluster_n=1), 2),
    (dict(in_format="nvfp4", out_format="e4m3"), 2),   # not on the pages
    (dict(n=96, epilogue="geglu"), 1),          # GeGLU pairs 32-column blocks too
    (dict(glu_limit=-1.0, epilogue="swiglu"), 1),
    (dict(glu_limit=float("inf"), epilogue="geglu"), 1),
    (dict(glu_alpha=float("nan"), epilogue="swiglu"), 1),
    (dict(glu_limit=7.0, epilogue="gate"), 1),  # GLU options belong to the GLUs
    (dict(glu_alpha=2.0, epilogue="srelu"), 1),
    # C is bf16 or f16 (with MXFP8 inputs also f32, e4m3, e5m2, e2m1)
    (dict(c_format="f32", in_format="nvfp4"), 1), (dict(c_format_code=3, in_format="mxfp4"), 1),
    (dict(c_format_code=6), 1),
    (dict(bias_format="e4m3"), 1), (dict(bias_format_code=9), 1),
    (dict(want_c_raw=2), 1),
    (dict(discrete_raw=2), 1),
    (dict(epilogue="dswiglu", c_format="bf16"), 1),      # the backward stores no C
    (dict(epilogue="dswiglu", bias_format="f32"), 1),    # and adds no bias
    (dict(epilogue="dswiglu", saved_c_format="e4m3"), 1),
    (dict(epilogue="dswiglu", n=80), 1),
    (dict(epilogue="dswiglu", tanh_clamp_s=4.0), 1),
    (dict(rht_format="e4m3"), 1), (dict(rht_format="f16"), 1),   # RHT is bf16 or NVFP4
    (dict(epilogue="dswiglu", rht_format="bf16"), 1),            # forward epilogues only
    (dict(epilogue="dswiglu", dgeglu_params=(1.0, -7.0, 7.0, 1.0)), 1),   # dGeGLU's own
    (dict(epilogue="dgeglu", dgeglu_params=(1.0, 7.0, -7.0, 1.0)), 1),    # min <= max
    (dict(epilogue="dgeglu", dgeglu_params=(float("nan"), -7.0, 7.0, 1.0)), 1),
    (dict(epilogue="dsituglu", situ_betas=(-1.0, 1.0)), 1),
    (dict(rht_format="bf16", rht_colwise=True), 1),               # colwise RHT is NVFP4
    (dict(n=128, epilogue="swiglu", rht_format="e2m1", rht_colwise=True), 1),   # N_out % 128
    (dict(epilogue="dsituglu", situ_betas=(1.0, float("inf"))), 1),
    (dict(epilogue="dswiglu", situ_betas=(2.0, 2.0)), 1),          # dSiTU-GLU's own
    # UE8M0-scaled FP4: (2, 1) clusters only as CTA pairs; no FP8 outputs from FP4
    (dict(in_format="mxfp4", tile_m=128, tile_n=256, cluster_m=2, cluster_n=1), 2),
    (dict(in_format="fp4_ue8m0_16", tile_m=128, tile_n=256, cluster_m=2, cluster_n=1), 2),
    (dict(in_format="mxfp4", out_format="e5m2"), 2),
    (dict(in_format="mxfp4", k=48), 1),                           # K % 32 for packed FP4
    # the BF16 backend: dSwiGLU / dGeGLU (fixed constants), 16/32-bit D, K % 8
    (dict(in_format="bf16"), 1),                                  # no forward epilogues
    (dict(in_format="bf16", epilogue="dsituglu"), 1),
    (dict(in_format="bf16", epilogue="dgeglu", dgeglu_params=(1.0, -7.0, 7.0, 1.0)), 1),
    (dict(in_format="bf16", epilogue="dswiglu", out_format="e4m3"), 1),
    (dict(in_format="bf16", epilogue="dswiglu", k=252), 1),
    (dict(in_format="bf16", epilogue="dswiglu", tile_m=128, tile_n=256, cluster_m=2, cluster_n=1), 2),
])
def test_create_rejects(lib, over, code):
    assert _create(**over) == code


@pytest.mark.parametrize("over", [
    dict(epilogue="geglu", n=128, glu_limit=7.0, glu_alpha=1.5),
    dict(epilogue="swiglu", glu_alpha=1.0, c_format="bf16", bias_format="f32"),
    dict(epilogue="srelu", glu_alpha=0.0, c_format="f16", bias_format="bf16"),
    dict(epilogue="gate", c_format="f32"), dict(epilogue="swiglu", c_format="e4m3"),
    dict(epilogue="srelu", c_format="e2m1", in_format="mxfp8_e5m2"),
    dict(epilogue="gate", bias_format="f16"),
    dict(discrete_b=True, num_groups=1024),
    dict(epilogue="dswiglu", n=96, saved_c_format="f32", out_format="e4m3", want_col=1),
    dict(epilogue="swiglu", rht_format="e2m1", in_format="nvfp4", out_format="e2m1"),
    dict(epilogue="dgeglu", dgeglu_params=(1.0, -10.0, 10.0, 0.0)),
    dict(epilogue="dsituglu", situ_betas=(2.0, 0.5)),
    dict(in_format="mxfp4", epilogue="srelu", out_format="e2m1", want_col=1, tile_m=256, tile_n=256,
         cluster_m=2, cluster_n=1),
    dict(in_format="fp4_ue8m0_16", epilogue="dswiglu", out_format="bf16"),
    dict(in_format="bf16", epilogue="dswiglu", out_format="f32", k=264),
    dict(in_format="bf16", epilogue="dgeglu", out_format="bf16", tile_m=256, tile_n=256, cluster_m=2,
         cluster_n=1, discrete_b=True),
])
def test_create_accepts_epilogue_options(lib, over):
    # validation passes: 0 with a GPU, else the device query that follows
    # validation fails with BSGG_ERR_CUDA
    assert _create(**over) in (0, 3)


def test_null_arguments(lib):
    assert lib.bsgg_create(None, None) == 1
    assert lib.bsgg_run(None, None, None) == 1
    assert lib.bsgg_query_device_status(None, None) == 1
    lib.bsgg_destroy(None)


def _struct_fields(name):
    src = open(HEADER).read()
    end = src.index("} " + name + ";")
    start = src.rindex("typedef struct {", 0, end)
    body = re.sub(r"/\*.*?\*/", "", src[start + len("typedef struct {"):end], flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?([A-Za-z0-9_]+)\s*(\*?)\s*([A-Za-z0-9_]+);", body, flags=re.M)


def test_binding_structs_match_the_header():
    """Field names, order and types of bsgg_desc and bsgg_args in the header
    equal the Python binding's ctypes structures (the ABI is positional)."""
    ctype = {"int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32, "float": ctypes.c_float}
    desc = _struct_fields("bsgg_desc")
    assert [n for _, _, n in desc] == [n for n, _ in bsgg.Desc._fields_]
    for (t, star, n), (pn, pt) in zip(desc, bsgg.Desc._fields_):
        assert star == "" and ctype[t] is pt, n
    args = _struct_fields("bsgg_args")
    assert [n for _, _, n in args] == [n for n, _ in bsgg.Args._fields_]
    assert all(star == "*" for _, star, _ in args)


def _enum_values(name):
    """{enumerator: value} of the header's typedef enum `name` (explicit values)."""
    src = open(HEADER).read()
    end = src.index("} " + name + ";")
    start = src.rindex("typedef enum {", 0, end)
    body = re.sub(r"/\*.*?\*/", "", src[start + len("typedef enum {"):end], flags=re.S)
    return {k: int(v) for k, v in re.findall(r"([A-Z0-9_]+)\s*=\s*(\d+)", body)}


def test_binding_enums_match_the_header():
    """The binding's format and epilogue names map to the header's values (the
    descriptor carries them as plain integers), and the generator knows every
    input format the binding does."""
    from block_scaled_grouped_gb300 import workloads as W
    ins = _enum_values("bsgg_in_format")
    assert ins == {"BSGG_IN_" + k.upper(): v for k, v in bsgg.IN_FORMATS.items()}
    outs = _enum_values("bsgg_out_format")
    assert outs == {"BSGG_OUT_" + k.upper(): v for k, v in bsgg.OUT_FORMATS.items()}
    epis = _enum_values("bsgg_epilogue")
    assert epis == {"BSGG_EPI_" + k.upper(): v for k, v in bsgg.EPILOGUES.items()}
    assert set(W.IN_FORMATS) == set(bsgg.IN_FORMATS)
    assert set(W.EPILOGUES) == set(bsgg.EPILOGUES) and set(W.BWD_EPILOGUES) == set(bsgg.BWD_EPILOGUES)


def test_noalloc_refuses_before_any_device_call(lib):
    """bsgg_run_noalloc validates the description first, exactly as
    bsgg_create does, and refuses what its static scratch cannot hold
    (discrete weight mode's per-expert tensor maps) before it touches a
    device; so these answers need no GPU."""
    import ctypes
    assert lib.bsgg_run_noalloc(None, None, None, 1) == 1
    args = bsgg.Args()
    for over, code in [(dict(m_pad=200), 1), (dict(num_groups=1025), 1),
                       (dict(n=96, epilogue="swiglu"), 1), (dict(discrete_b=True), 2)]:
        d = dict(m_pad=384, n=256, k=256, num_groups=2, in_format="mxfp8_e4m3", out_format="bf16",
                 epilogue="gate")
        d.update(over)
        desc = bsgg.make_desc(**d)
        assert lib.bsgg_run_noalloc(ctypes.byref(desc), ctypes.byref(args), None, 1) == code, over


def test_helper_entry_points_refuse_bad_arguments_before_any_device_call(lib):
    """The helpers check their arguments on the host first, as the header
    states, so these refusals need no GPU."""
    import ctypes
    out = ctypes.c_double(0.0)
    # packer: null buffers, empty extents
    assert lib.bsgg_pack_sf(None, None, 128, 4, 1, None) == 1
    dummy = ctypes.c_void_p(16)          # never dereferenced: the extents are refused first
    for rows, kb, sl in [(0, 4, 1), (128, 0, 1), (128, 4, 0), (-1, 4, 1)]:
        assert lib.bsgg_pack_sf(dummy, dummy, rows, kb, sl, None) == 1
    # scale-factor sizes of empty extents are 0
    assert lib.bsgg_sf_bytes(0, 256, 32, 1) == 0 and lib.bsgg_sf_bytes(128, 256, 0, 1) == 0
    # MMA-rate measurement: output pointer, tile_n, instruction count, input format
    assert lib.bsgg_measure_mma_peak(0, 128, 1024, None, None) == 1
    for fmt, tn, cnt in [(0, 192, 1024), (0, 128, 3), (0, 128, (1 << 22) + 1), (5, 128, 1024), (-1, 256, 1024)]:
        assert lib.bsgg_measure_mma_peak(fmt, tn, cnt, ctypes.byref(out), None) == 1
    # the same for either instruction form: tile_m 128 or 256, pairs 256 x 256 only
    assert lib.bsgg_measure_mma_peak_tile(0, 256, 256, 1024, None, None) == 1
    for fmt, tm, tn, cnt in [(0, 64, 256, 1024), (0, 512, 256, 1024), (0, 256, 192, 1024), (0, 256, 256, 3),
                             (2, 256, 256, (1 << 22) + 1), (5, 256, 256, 1024)]:
        assert lib.bsgg_measure_mma_peak_tile(fmt, tm, tn, cnt, ctypes.byref(out), None) == 1
    assert lib.bsgg_measure_mma_peak_tile(0, 256, 128, 1024, ctypes.byref(out), None) == 2
    # plan-taking entry points with no plan
    assert lib.bsgg_run_host(None, None, None, None, None, None) == 1
    assert lib.bsgg_run_host_async(None, None, None, None, None, None) == 1
    assert lib.bsgg_debug_force_timeout(None, 1) == 1
    assert lib.bsgg_launches_per_run(None) == -1
