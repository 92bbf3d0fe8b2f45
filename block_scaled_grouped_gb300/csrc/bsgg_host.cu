// bsgg_host.cu -- the C ABI declared in include/bsgg.h: validation (the pages'
// "Support Surface and Constraints"), plan creation, TMA descriptor encoding,
// kernel launch, the device status word, the scale-factor packer and the
// host-buffer end-to-end call.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <algorithm>
#include <new>

#include "../../include/bsgg.h"
#include "bsgg_internal.h"

struct bsgg_plan {
  bsgg_desc desc;
  int device;
  int num_sms;
  int grid;                // CTAs per launch (a multiple of 2 for clusters)
  bool pair;               // 256 x 256 tiles on CTA pairs (2-CTA MMAs)
  int ic;                  // the kernel's input class (bsgg::IC_*)
  int slices;              // 128-byte K slices per pipeline stage (bsgg::stage_slices)
  int bn;
  int epi;
  int outc;
  int sf_vec;
  int64_t kbytes;          // bytes per row of A / B
  int64_t n_out;
  int64_t out_row_bytes;
  uint32_t* status;        // device word: kStatus* bits
  bool force_timeout;      // bsgg_debug_force_timeout
  int32_t dbg_margin;      // bsgg_debug_bounds_margin (range-checking build)
  uint32_t violation[3];   // the last range-check failure read back: site, value, limit
  CUtensorMap* maps;       // discrete weight mode: {B_g, SFB_g} per expert, then the bad-pointer flag
};

namespace {

using bsgg::Launch;

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Barrier-wait bound while bsgg_debug_force_timeout is on: short, so that the
// test's launch ends quickly.
constexpr uint64_t kTestWaitLimitNs = 50000000ull;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

uint64_t sf_bytes_impl(int64_t rows, int64_t cols, int64_t v, int64_t L) {
  return static_cast<uint64_t>(512) * L * ceil_div(rows, 128) * ceil_div(ceil_div(cols, v), 4);
}

bool is_quant(int out) { return out == BSGG_OUT_E4M3 || out == BSGG_OUT_E5M2 || out == BSGG_OUT_E2M1; }

// The backward epilogues ("Grouped GEMM + dGLU (SM100)"): GEMM scaled by alpha^2,
// the saved C read, D twice as wide as the GEMM, dprob accumulated.
bool is_bwd_epi(int epi) {
  return epi == BSGG_EPI_DSWIGLU || epi == BSGG_EPI_DGEGLU || epi == BSGG_EPI_DSITUGLU;
}

int out_elem_bits(int out) {
  switch (out) {
    case BSGG_OUT_BF16: case BSGG_OUT_F16: return 16;
    case BSGG_OUT_F32: return 32;
    case BSGG_OUT_E4M3: case BSGG_OUT_E5M2: return 8;
    default: return 4;
  }
}

// FP4 data (E2M1) with E4M3 or UE8M0 scales; the UE8M0-scaled ones; bfloat16
// operands without scales (the BF16 backend of the dGLU backward)
bool is_fp4_in(int f) { return f == BSGG_IN_NVFP4 || f == BSGG_IN_FP4_UE8M0_16 || f == BSGG_IN_MXFP4; }
bool is_f4e8_in(int f) { return f == BSGG_IN_FP4_UE8M0_16 || f == BSGG_IN_MXFP4; }

bsgg_status validate(const bsgg_desc* d) {
  if (!d) return BSGG_ERR_INVALID_ARG;
  // tile shape: the pages' mma_tiler_mn with TILE_M in {128, 256} (256 = 2-CTA
  // instructions) and TILE_N in {128, 256}; pairs are built for 256 x 256 only
  if (d->tile_m != 0 && d->tile_m != 128 && d->tile_m != 256) return BSGG_ERR_INVALID_ARG;
  if (d->tile_n != 0 && d->tile_n != 128 && d->tile_n != 256) return BSGG_ERR_INVALID_ARG;
  if (d->tile_m == 256 && d->tile_n == 128) return BSGG_ERR_UNSUPPORTED;
  // cluster shape: the pages' cluster_shape_mn, powers of two <= 4 (both or
  // neither given); 2-CTA tiles need an even CLUSTER_M ("Grouped GEMM + Quant
  // (SM100)", Tiling and Cluster).  Built: (1, 1) with 128-row tiles and
  // (2, 1) with 256 x 256 tiles (the CTA pair).  A (2, 1) cluster of 128-row
  // tiles would share an operand tile between the two CTAs by TMA multicast;
  // this library issues no multicast loads, so it is refused.
  auto pow2le4 = [](int v) { return v == 1 || v == 2 || v == 4; };
  if ((d->cluster_m == 0) != (d->cluster_n == 0)) return BSGG_ERR_INVALID_ARG;
  if (d->cluster_m != 0) {
    if (!pow2le4(d->cluster_m) || !pow2le4(d->cluster_n)) return BSGG_ERR_INVALID_ARG;
    if (d->tile_m == 256 && d->cluster_m % 2 != 0) return BSGG_ERR_INVALID_ARG;
    if (d->cluster_n != 1 || d->cluster_m > 2) return BSGG_ERR_UNSUPPORTED;
    if (d->cluster_m == 2 && (d->tile_m == 128 || d->tile_n == 128)) return BSGG_ERR_UNSUPPORTED;
  }
  if (d->num_groups < 1 || d->num_groups > 1024) return BSGG_ERR_INVALID_ARG;   // L <= 1024
  if (d->m_pad <= 0 || d->m_pad % 128 != 0 || d->m_pad > (int64_t(1) << 30)) return BSGG_ERR_INVALID_ARG;
  if (d->n <= 0 || d->k <= 0 || d->n > (int64_t(1) << 24) || d->k > (int64_t(1) << 24))
    return BSGG_ERR_INVALID_ARG;
  if (d->in_format < BSGG_IN_MXFP8_E4M3 || d->in_format > BSGG_IN_BF16) return BSGG_ERR_INVALID_ARG;
  if (d->out_format < BSGG_OUT_BF16 || d->out_format > BSGG_OUT_E2M1) return BSGG_ERR_INVALID_ARG;
  if (d->epilogue < BSGG_EPI_GATE || d->epilogue > BSGG_EPI_DSITUGLU) return BSGG_ERR_INVALID_ARG;
  const bool glu = d->epilogue == BSGG_EPI_SWIGLU || d->epilogue == BSGG_EPI_GEGLU;
  const bool bwd = is_bwd_epi(d->epilogue);
  // dSiTU-GLU's tanh scales: finite, > 0 (0 = 1); nothing else reads them
  if (!std::isfinite(d->situ_beta1) || !std::isfinite(d->situ_beta2) || d->situ_beta1 < 0.0f ||
      d->situ_beta2 < 0.0f || (d->epilogue != BSGG_EPI_DSITUGLU && (d->situ_beta1 != 0.0f || d->situ_beta2 != 0.0f)))
    return BSGG_ERR_INVALID_ARG;
  if (d->dgeglu_custom != 0 && d->dgeglu_custom != 1) return BSGG_ERR_INVALID_ARG;
  if (d->dgeglu_custom &&
      (d->epilogue != BSGG_EPI_DGEGLU || !std::isfinite(d->dgeglu_alpha) || !std::isfinite(d->dgeglu_clamp_min) ||
       !std::isfinite(d->dgeglu_clamp_max) || !std::isfinite(d->dgeglu_linear_offset) ||
       d->dgeglu_clamp_min > d->dgeglu_clamp_max))
    return BSGG_ERR_INVALID_ARG;
  if (d->gate_first != 0 && d->gate_first != 1) return BSGG_ERR_INVALID_ARG;
  if (d->want_col != 0 && d->want_col != 1) return BSGG_ERR_INVALID_ARG;
  // K-major rows must be 16-byte aligned ("Support Surface and Constraints",
  // Layouts and Strides): K % 16 for FP8, K % 32 for packed FP4, K % 8 for bf16.
  const bool fp4 = is_fp4_in(d->in_format), bf16_in = d->in_format == BSGG_IN_BF16;
  if (d->k % (fp4 ? 32 : bf16_in ? 8 : 16) != 0) return BSGG_ERR_INVALID_ARG;
  // The BF16 backend ("Grouped GEMM + dGLU (SM100)", Backend dispatch and BF16
  // contract): dSwiGLU and dGeGLU with the source GeGLU constants, 16/32-bit
  // D_row, no D_col, scale factors or norm_const
  if (bf16_in && ((d->epilogue != BSGG_EPI_DSWIGLU && d->epilogue != BSGG_EPI_DGEGLU) || d->dgeglu_custom ||
                  is_quant(d->out_format)))
    return BSGG_ERR_INVALID_ARG;
  // SwiGLU pairs 32-column blocks: N % 64 ("Grouped GEMM + SwiGLU (SM100)",
  // Shapes and Divisibility).  Outputs are written in 32-column chunks.
  if (glu ? (d->n % 64 != 0) : (d->n % 32 != 0)) return BSGG_ERR_INVALID_ARG;
  if (!(std::isfinite(d->tanh_clamp_s) && d->tanh_clamp_s >= 0.0f)) return BSGG_ERR_INVALID_ARG;
  if (d->tanh_clamp_s > 0.0f && d->epilogue != BSGG_EPI_SRELU) return BSGG_ERR_INVALID_ARG;
  // glu_limit and glu_alpha belong to the GLUs ("Grouped GEMM + GLU + Hadamard +
  // Quant (SM100)", Configuration); 0 leaves either unset
  if (!(std::isfinite(d->glu_limit) && d->glu_limit >= 0.0f) || !std::isfinite(d->glu_alpha))
    return BSGG_ERR_INVALID_ARG;
  if (!glu && (d->glu_limit != 0.0f || (d->glu_alpha != 0.0f && d->glu_alpha != 1.0f)))
    return BSGG_ERR_INVALID_ARG;
  // C is stored as float16 or bfloat16; the bias is float16, bfloat16 or float32
  // ("Grouped GEMM + GLU + Hadamard + Quant (SM100)", Input/output tensors)
  if (d->want_c != 0 && d->want_c != 1) return BSGG_ERR_INVALID_ARG;
  // C with FP8 inputs may also be float32, float8_e4m3fn, float8_e5m2 or
  // float4_e2m1fn_x2 ("Grouped GEMM + SwiGLU (SM100)" and "Grouped GEMM + sReLU
  // (SM100)", output tensor C; no scale factor: a saturating conversion)
  if (d->want_c && d->c_format != BSGG_OUT_BF16 && d->c_format != BSGG_OUT_F16 &&
      !(d->in_format <= BSGG_IN_MXFP8_E5M2 && d->c_format >= BSGG_OUT_F32 && d->c_format <= BSGG_OUT_E2M1))
    return BSGG_ERR_INVALID_ARG;
  if (d->want_bias != 0 && d->want_bias != 1) return BSGG_ERR_INVALID_ARG;
  if (d->want_bias && d->bias_format != BSGG_OUT_BF16 && d->bias_format != BSGG_OUT_F16 &&
      d->bias_format != BSGG_OUT_F32)
    return BSGG_ERR_INVALID_ARG;
  if (d->discrete_b != 0 && d->discrete_b != 1) return BSGG_ERR_INVALID_ARG;
  // the dSwiGLU backward reads the saved C (bf16, f16 or f32); it adds no bias
  // and stores no C of its own
  if (bwd && (d->want_c || d->want_bias)) return BSGG_ERR_INVALID_ARG;
  if (bwd && d->saved_c_format != BSGG_OUT_BF16 && d->saved_c_format != BSGG_OUT_F16 &&
      d->saved_c_format != BSGG_OUT_F32)
    return BSGG_ERR_INVALID_ARG;
  // the Hadamard output: bf16 or NVFP4, forward epilogues only
  if (d->want_rht < 0 || d->want_rht > 2) return BSGG_ERR_INVALID_ARG;
  if (d->want_rht && ((d->rht_format != BSGG_OUT_BF16 && d->rht_format != BSGG_OUT_E2M1) || bwd))
    return BSGG_ERR_INVALID_ARG;
  // colwise: NVFP4 only, N_out % 128 (per-expert scale segments of N_out * expert_m / 16
  // bytes; "Grouped GEMM + GLU + Hadamard + Quant (SM100)", Constraints)
  if (d->want_rht == 2) {
    const int64_t n_out = glu ? d->n / 2 : d->n;
    if (d->rht_format != BSGG_OUT_E2M1 || n_out % 128 != 0) return BSGG_ERR_INVALID_ARG;
  }
  if (d->want_col && !is_quant(d->out_format)) return BSGG_ERR_INVALID_ARG;
  // NVFP4 inputs: the pages allow 16/32-bit float outputs; FP4 output is this
  // build's reading for the NVFP4 sReLU workload.  FP8 outputs from FP4 inputs
  // are not on the pages.
  if (fp4 && (d->out_format == BSGG_OUT_E4M3 || d->out_format == BSGG_OUT_E5M2)) return BSGG_ERR_UNSUPPORTED;
  return BSGG_OK;
}

uint32_t make_idesc(int in_format, int bn, bool pair) {
  uint32_t fmt, scale_ue8m0;
  if (in_format == BSGG_IN_BF16) {
    // kind::f16: F32 accumulator (bits 4-5 = 1), BF16 A and B (format 1)
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(bn >> 3) << 17) |
           (static_cast<uint32_t>((pair ? 2 * bsgg::kBM : bsgg::kBM) >> 4) << 24);
  }
  if (in_format == BSGG_IN_NVFP4) { fmt = 1; scale_ue8m0 = 0; }          // E2M1, UE4M3 scales
  else if (is_f4e8_in(in_format)) { fmt = 1; scale_ue8m0 = 1; }       // E2M1, UE8M0 scales (per 16 slots)
  else { fmt = (in_format == BSGG_IN_MXFP8_E4M3) ? 0u : 1u; scale_ue8m0 = 1; }  // E4M3/E5M2, UE8M0
  uint32_t d = 0;
  d |= fmt << 7;                                      // A format
  d |= fmt << 10;                                     // B format
  d |= static_cast<uint32_t>(bn >> 3) << 17;          // N / 8
  d |= scale_ue8m0 << 23;                             // scale format
  d |= static_cast<uint32_t>((pair ? 2 * bsgg::kBM : bsgg::kBM) >> 4) << 24;   // M / 16
  return d;                                           // both operands K-major, no negation
}

bsgg_status encode_one(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto enc = get_encode_fn();
  if (!enc) return BSGG_ERR_CUDA;
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                         dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSGG_OK : BSGG_ERR_CUDA;
}

// A (m_pad, K bytes) and B (L, N, K bytes) as 128-byte-swizzled boxes of
// 128 K-bytes x 128 rows / x (rows of B one load moves: the tile's, half of it
// in a CTA pair); the scale factors as
// (256 bytes, 2 * atoms, 128-row blocks) so that one box moves a stage's
// 512-byte atoms of one (SFA) or two (SFB, tile_n = 256) row blocks.
bsgg_status encode_maps(const bsgg_plan* P, const bsgg_args* a, bsgg::Launch* L) {
  const bsgg_desc& d = P->desc;
  const int64_t kq = ceil_div(ceil_div(d.k, P->sf_vec), 4);
  // scale atoms per stage (an atom = 4 scales of 128 rows): per 128-byte K
  // slice 4 for FP4 with one scale per 16 values, 2 per 32, 1 for MXFP8
  const bool fp4 = is_fp4_in(P->desc.in_format);
  const int atoms = (!fp4 ? 1 : P->sf_vec == 32 ? 2 : 4) * P->slices;
  bsgg_status st;
  {
    cuuint64_t dims[2] = {cuuint64_t(P->kbytes), cuuint64_t(d.m_pad)};
    cuuint64_t strides[1] = {cuuint64_t(P->kbytes)};
    cuuint32_t box[2] = {bsgg::kBKBytes, cuuint32_t(bsgg::kBM)};
    if ((st = encode_one(&L->tmA, a->a, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != BSGG_OK) return st;
  }
  // discrete weight mode: B and SFB maps of one expert (one slice) whose global
  // address, a placeholder here (the plan's own workspace), is replaced per
  // expert on the device
  const bool disc = d.discrete_b != 0;
  const int64_t slices = disc ? 1 : d.num_groups;
  const void* b_base = disc ? static_cast<const void*>(P->maps) : a->b;
  const void* sfb_base = disc ? static_cast<const void*>(P->maps) : a->sfb;
  {
    cuuint64_t dims[3] = {cuuint64_t(P->kbytes), cuuint64_t(d.n), cuuint64_t(slices)};
    cuuint64_t strides[2] = {cuuint64_t(P->kbytes), cuuint64_t(P->kbytes * d.n)};
    cuuint32_t box[3] = {bsgg::kBKBytes, cuuint32_t(P->pair ? P->bn / 2 : P->bn), 1};
    if ((st = encode_one(&L->tmB, b_base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != BSGG_OK)
      return st;
  }
  // bfloat16 operands have no scale factors: the scale maps stay zero (unused)
  if (d.in_format == BSGG_IN_BF16) {
    std::memset(&L->tmSFA, 0, sizeof(L->tmSFA));
    std::memset(&L->tmSFB, 0, sizeof(L->tmSFB));
    return BSGG_OK;
  }
  {
    cuuint64_t dims[3] = {256, cuuint64_t(2 * kq), cuuint64_t(ceil_div(d.m_pad, 128))};
    cuuint64_t strides[2] = {256, cuuint64_t(512 * kq)};
    cuuint32_t box[3] = {256, cuuint32_t(2 * atoms), 1};
    if ((st = encode_one(&L->tmSFA, a->sfa, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != BSGG_OK)
      return st;
  }
  {
    cuuint64_t dims[3] = {256, cuuint64_t(2 * kq), cuuint64_t(ceil_div(d.n, 128) * slices)};
    cuuint64_t strides[2] = {256, cuuint64_t(512 * kq)};
    cuuint32_t box[3] = {256, cuuint32_t(2 * atoms), cuuint32_t(P->bn / 128)};
    if ((st = encode_one(&L->tmSFB, sfb_base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != BSGG_OK)
      return st;
  }
  return BSGG_OK;
}

// D and D_col as byte tensors (row bytes, m_pad) whose boxes are one warp's
// 32-row chunk (32 values: 64 bytes of bf16/f16, 32 of FP8, 16 of packed FP4),
// stored by the epilogue through TMA; fp32 D is stored directly (zero maps).
bsgg_status encode_out_maps(const bsgg_plan* P, const bsgg_args* a, bsgg::Launch* L) {
  const bsgg_desc& d = P->desc;
  std::memset(&L->tmD, 0, sizeof(L->tmD));
  std::memset(&L->tmDcol, 0, sizeof(L->tmDcol));
  if (d.out_format == BSGG_OUT_F32) return BSGG_OK;
  const cuuint32_t chunk = static_cast<cuuint32_t>(32 * out_elem_bits(d.out_format) / 8);
  cuuint64_t dims[2] = {cuuint64_t(P->out_row_bytes), cuuint64_t(d.m_pad)};
  cuuint64_t strides[1] = {cuuint64_t(P->out_row_bytes)};
  cuuint32_t box[2] = {chunk, 32};
  bsgg_status st = encode_one(&L->tmD, a->d, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st == BSGG_OK && d.want_col)
    st = encode_one(&L->tmDcol, a->d_col, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  return st;
}

// Everything a plan derives from its description and the current device.
bsgg_status init_plan(const bsgg_desc* desc, int device, int num_sms, bsgg_plan* P) {
  P->desc = *desc;
  P->device = device;
  P->num_sms = num_sms;
  // library choice (measured on GB300): 256 x 256 tiles on CTA pairs (half
  // the shared-memory operand traffic per MMA of 1-CTA tiles): MXFP8 FC1
  // 2741-2779 vs 2608-2655 TFLOP/s for 128 x 256, NVFP4 fine-grained
  // 4937-4985 vs 4859-4907 (three alternating bench runs each)
  // The dSwiGLU backward writes four outputs per accumulator value and reads
  // two saved values: with 128-column tiles its epilogue holds half the
  // accumulator columns per thread and runs without register spills (measured
  // on GB300: 1418 TFLOP/s on the FC1 backward against 582 with 256 x 256
  // pairs, whose epilogue spills to local memory).
  // The bfloat16 backward (no scale slots in tensor memory) holds two 256-column
  // accumulators and reads them 32 columns at a time: pairs measured 1371
  // TFLOP/s on the FC1 backward against 1215 for 128 x 256 and 907 for 128 x 128.
  const bool bwd = is_bwd_epi(desc->epilogue);
  const bool pair_default = !bwd || desc->in_format == BSGG_IN_BF16;
  // a (2, 1) cluster is always a CTA pair (validation refuses it with 128-row
  // or 128-column tiles)
  int tm = desc->tile_m, tn = desc->tile_n;
  const int cm = desc->cluster_m;
  if (tm == 0) tm = (cm == 2 || (tn != 128 && cm != 1 && pair_default)) ? 256 : 128;
  if (tn == 0) tn = (bwd && tm == 128) ? 128 : 256;
  P->pair = (tm == 256);
  P->bn = P->pair ? 256 : tn;
  P->ic = desc->in_format == BSGG_IN_BF16    ? bsgg::IC_BF16
          : desc->in_format == BSGG_IN_NVFP4 ? bsgg::IC_NVF4
          : is_f4e8_in(desc->in_format)      ? bsgg::IC_F4E8
                                             : bsgg::IC_MXF8;
  P->slices = bsgg::stage_slices(P->ic, P->pair ? bsgg::CM_PAIR : bsgg::CM_SINGLE);
  // GeGLU runs in the SwiGLU instances (Params::glu_kind selects the activation)
  // the dGeGLU backward runs in the dSwiGLU instances (Params::bwd_kind)
  P->epi = desc->epilogue == BSGG_EPI_GEGLU ? bsgg::EPI_SWIGLU
           : desc->epilogue == BSGG_EPI_DSITUGLU ? bsgg::EPI_DSITUGLU
           : is_bwd_epi(desc->epilogue)     ? bsgg::EPI_DSWIGLU
                                            : desc->epilogue;
  P->outc = desc->out_format == BSGG_OUT_E2M1 ? bsgg::OUTC_FP4
            : is_quant(desc->out_format)      ? bsgg::OUTC_FP8
                                              : bsgg::OUTC_FLOAT;
  const bool fp4 = is_fp4_in(desc->in_format);
  P->sf_vec = (desc->in_format == BSGG_IN_NVFP4 || desc->in_format == BSGG_IN_FP4_UE8M0_16) ? 16 : 32;
  P->kbytes = fp4 ? desc->k / 2 : desc->in_format == BSGG_IN_BF16 ? 2 * desc->k : desc->k;
  P->n_out = (desc->epilogue == BSGG_EPI_SWIGLU || desc->epilogue == BSGG_EPI_GEGLU) ? desc->n / 2
             : is_bwd_epi(desc->epilogue)                                             ? 2 * desc->n
                                                                                      : desc->n;
  P->out_row_bytes = P->n_out * out_elem_bits(desc->out_format) / 8;
  if (P->pair) {
    int resident = bsgg::cluster_resident_ctas(fp4);
    if (resident <= 0) resident = num_sms;
    P->grid = std::max(2, (std::min(resident, num_sms) / 2) * 2);
  } else {
    P->grid = num_sms;
  }
  return BSGG_OK;
}

bsgg_status check_args(const bsgg_plan* P, const bsgg_args* a) {
  if (!a) return BSGG_ERR_INVALID_ARG;
  const bsgg_desc& d = P->desc;
  // bfloat16 operands take no scale factors (sfa, sfb and sfb_ptrs are not read)
  const bool scaled = d.in_format != BSGG_IN_BF16;
  const void* need[] = {a->a, scaled ? a->sfa : a->a, a->padded_offsets, a->alpha, a->prob, a->d};
  for (const void* p : need)
    if (!p || !aligned16(p)) return BSGG_ERR_INVALID_ARG;
  // dense and discrete weights are mutually exclusive ("Grouped GEMM + GLU +
  // Hadamard + Quant (SM100)", Constraints)
  if (d.discrete_b) {
    if (a->b || a->sfb || !a->b_ptrs || !aligned16(a->b_ptrs)) return BSGG_ERR_INVALID_ARG;
    if (scaled && (!a->sfb_ptrs || !aligned16(a->sfb_ptrs))) return BSGG_ERR_INVALID_ARG;
  } else {
    if (a->b_ptrs || a->sfb_ptrs || !a->b || !aligned16(a->b)) return BSGG_ERR_INVALID_ARG;
    if (scaled && (!a->sfb || !aligned16(a->sfb))) return BSGG_ERR_INVALID_ARG;
  }
  if (is_quant(d.out_format)) {
    if (!a->sfd_row || !a->norm_const || !aligned16(a->sfd_row)) return BSGG_ERR_INVALID_ARG;
    if (d.want_col && (!a->d_col || !a->sfd_col || !aligned16(a->d_col) || !aligned16(a->sfd_col)))
      return BSGG_ERR_INVALID_ARG;
  } else if (d.out_format != BSGG_OUT_F32 && scaled && !a->amax) {
    return BSGG_ERR_INVALID_ARG;   // amax required for bf16/f16 D (optional on the BF16 backend)
  }
  if (d.want_bias && (!a->bias || !aligned16(a->bias))) return BSGG_ERR_INVALID_ARG;
  if (d.epilogue == BSGG_EPI_DSWIGLU && (!a->saved_c || !aligned16(a->saved_c) || !a->beta || !a->dprob))
    return BSGG_ERR_INVALID_ARG;
  if ((d.epilogue == BSGG_EPI_DGEGLU || d.epilogue == BSGG_EPI_DSITUGLU) &&
      (!a->saved_c || !aligned16(a->saved_c) || !a->dprob))
    return BSGG_ERR_INVALID_ARG;
  // the BF16 contract scales C by beta for dGeGLU too (X = beta C)
  if (!scaled && d.epilogue == BSGG_EPI_DGEGLU && !a->beta) return BSGG_ERR_INVALID_ARG;
  if (d.want_rht && (!a->rht || !aligned16(a->rht))) return BSGG_ERR_INVALID_ARG;
  if (a->dbias && !is_bwd_epi(d.epilogue)) return BSGG_ERR_INVALID_ARG;   // a backward output
  if (d.want_rht && d.rht_format == BSGG_OUT_E2M1 && (!a->sfrht || !a->rht_norm_const))
    return BSGG_ERR_INVALID_ARG;
  if (d.want_c && (!a->c || !aligned16(a->c))) return BSGG_ERR_INVALID_ARG;
  return BSGG_OK;
}

__global__ void pack_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows,
                               int64_t kblocks, int64_t R, int64_t KQ, int64_t total) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    // physical order (l, row-block, k-atom, row%32, (row/32)%4, kblk%4)
    const int64_t k4 = i & 3, r4 = (i >> 2) & 3, r32 = (i >> 4) & 31;
    int64_t rest = i >> 9;
    const int64_t ka = rest % KQ;
    rest /= KQ;
    const int64_t rb = rest % R;
    const int64_t l = rest / R;
    const int64_t row = rb * 128 + r4 * 32 + r32, kb = ka * 4 + k4;
    dst[i] = (row < rows && kb < kblocks) ? src[(l * rows + row) * kblocks + kb] : uint8_t(0);
  }
}

// Discrete weight mode: expert g's maps are the templates with the global
// address replaced by b_ptrs[g] / sfb_ptrs[g].  One block, one thread per
// expert.  An expert that owns rows needs both pointers non-null and 16-byte
// aligned; otherwise the flag after the maps is raised (the GEMM then writes
// nothing) along with the status bit.  Experts without rows keep the
// placeholder address; their maps are never used.  Without scale factors
// (bfloat16 operands, scaled = 0) sfb_ptrs is not read and the scale maps are
// left as the (unused) template.
__global__ void expert_maps_kernel(const __grid_constant__ CUtensorMap tB, const __grid_constant__ CUtensorMap tSFB,
                                   const int64_t* __restrict__ b_ptrs, const int64_t* __restrict__ sfb_ptrs,
                                   int scaled, const int32_t* __restrict__ offsets, int L, CUtensorMap* maps,
                                   uint32_t* status) {
  const int g = threadIdx.x;
  int bad = 0;
  if (g < L) {
    const int32_t start = g ? offsets[g - 1] : 0;
    const bool used = offsets[g] != start;
    const uint64_t pb = static_cast<uint64_t>(b_ptrs[g]);
    const uint64_t ps = scaled ? static_cast<uint64_t>(sfb_ptrs[g]) : 16u;
    maps[2 * g] = tB;
    maps[2 * g + 1] = tSFB;
    if (used) {
      if (pb == 0 || ps == 0 || (pb & 15u) != 0 || (ps & 15u) != 0) {
        bad = 1;
      } else {
        bsgg::tmap_replace_address(&maps[2 * g], pb);
        if (scaled) bsgg::tmap_replace_address(&maps[2 * g + 1], ps);
      }
    }
    bsgg::tmap_release();
  }
  bad = __syncthreads_or(bad);
  if (g == 0) {
    *reinterpret_cast<uint32_t*>(maps + 2 * L) = bad ? 1u : 0u;
    if (bad) atomicOr(status, bsgg::kStatusBadPointers);
  }
}

// Bytes of the discrete-mode workspace: two maps per expert and a flag word.
size_t maps_bytes(int L) { return sizeof(CUtensorMap) * (2 * size_t(L) + 1); }

// The status a device status word stands for.  A bit this library does not
// define (it never writes one) reads as a CUDA error rather than as success.
bsgg_status status_of_word(uint32_t w) {
  if (w & bsgg::kStatusBounds) return BSGG_ERR_DEVICE_BOUNDS;
  if (w & bsgg::kStatusBadPointers) return BSGG_ERR_BAD_POINTERS;
  if (w & bsgg::kStatusBadOffsets) return BSGG_ERR_BAD_OFFSETS;
  if (w & bsgg::kStatusTimeout) return BSGG_ERR_DEVICE_TIMEOUT;
  return w == 0 ? BSGG_OK : BSGG_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* bsgg_status_string(bsgg_status s) {
  switch (s) {
    case BSGG_OK: return "ok";
    case BSGG_ERR_INVALID_ARG: return "invalid argument";
    case BSGG_ERR_UNSUPPORTED: return "unsupported configuration";
    case BSGG_ERR_CUDA: return "CUDA error";
    case BSGG_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case BSGG_ERR_BAD_OFFSETS: return "padded_offsets invalid";
    case BSGG_ERR_BAD_POINTERS: return "expert weight pointer invalid";
    case BSGG_ERR_DEVICE_BOUNDS: return "an index failed its range check";
  }
  return "unknown status";
}

uint64_t bsgg_sf_bytes(int64_t rows, int64_t cols, int32_t sf_vec, int32_t num_slices) {
  if (rows <= 0 || cols <= 0 || sf_vec <= 0 || num_slices <= 0) return 0;
  return sf_bytes_impl(rows, cols, sf_vec, num_slices);
}

int64_t bsgg_sf_offset(int64_t row, int64_t kblk, int64_t l, int64_t rows, int64_t kblocks) {
  const int64_t R = ceil_div(rows, 128), KQ = ceil_div(kblocks, 4);
  return ((l * R + row / 128) * KQ + kblk / 4) * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4 + kblk % 4;
}

bsgg_status bsgg_pack_sf(const uint8_t* rowmajor, uint8_t* swizzled, int64_t rows, int64_t kblocks,
                         int32_t num_slices, void* stream) {
  if (!rowmajor || !swizzled || rows <= 0 || kblocks <= 0 || num_slices <= 0) return BSGG_ERR_INVALID_ARG;
  const int64_t R = ceil_div(rows, 128), KQ = ceil_div(kblocks, 4);
  const int64_t total = int64_t(num_slices) * R * KQ * 512;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>(ceil_div(total, threads), 4096);
  pack_sf_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      rowmajor, swizzled, rows, kblocks, R, KQ, total);
  return cudaGetLastError() == cudaSuccess ? BSGG_OK : BSGG_ERR_CUDA;
}

bsgg_status bsgg_create(const bsgg_desc* desc, bsgg_plan** plan) {
  if (!plan) return BSGG_ERR_INVALID_ARG;
  *plan = nullptr;
  const bsgg_status v = validate(desc);
  if (v != BSGG_OK) return v;
  bsgg_plan* P = new (std::nothrow) bsgg_plan();
  if (!P) return BSGG_ERR_INVALID_ARG;
  P->desc = *desc;
  if (cudaGetDevice(&P->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device) != cudaSuccess) {
    delete P;
    return BSGG_ERR_CUDA;
  }
  if (init_plan(desc, P->device, P->num_sms, P) != BSGG_OK) {
    delete P;
    return BSGG_ERR_CUDA;
  }
  if (cudaMalloc(&P->status, 16) != cudaSuccess) {
    delete P;
    return BSGG_ERR_CUDA;
  }
  if (cudaMemset(P->status, 0, 16) != cudaSuccess) {
    cudaFree(P->status);
    delete P;
    return BSGG_ERR_CUDA;
  }
  if (desc->discrete_b && cudaMalloc(&P->maps, maps_bytes(desc->num_groups)) != cudaSuccess) {
    cudaFree(P->status);
    delete P;
    return BSGG_ERR_CUDA;
  }
  *plan = P;
  return BSGG_OK;
}

void bsgg_destroy(bsgg_plan* plan) {
  if (!plan) return;
  if (plan->status) cudaFree(plan->status);
  if (plan->maps) cudaFree(plan->maps);
  delete plan;
}

bsgg_status bsgg_run(bsgg_plan* P, const bsgg_args* a, void* stream) {
  if (!P) return BSGG_ERR_INVALID_ARG;
  bsgg_status st = check_args(P, a);
  if (st != BSGG_OK) return st;
  const bsgg_desc& d = P->desc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch L;
  std::memset(&L, 0, sizeof(L));
  st = encode_maps(P, a, &L);
  if (st == BSGG_OK) st = encode_out_maps(P, a, &L);
  if (st != BSGG_OK) return st;
  // amax: one float per group, two for the backward (input / gate gradients)
  const int64_t n_amax = d.num_groups * (is_bwd_epi(d.epilogue) ? 2 : 1);
  if (a->amax && cudaMemsetAsync(a->amax, 0, sizeof(float) * n_amax, s) != cudaSuccess)
    return BSGG_ERR_CUDA;

  bsgg::Params& p = L.p;
  p.offsets = a->padded_offsets;
  p.alpha = a->alpha;
  p.prob = a->prob;
  p.norm_const = a->norm_const;
  p.d = a->d;
  p.d_col = a->d_col;
  p.sfd_row = static_cast<uint8_t*>(a->sfd_row);
  p.sfd_col = static_cast<uint8_t*>(a->sfd_col);
  p.amax = a->amax;
  p.status = P->status;
  p.m_pad = static_cast<int32_t>(d.m_pad);
  p.n = static_cast<int32_t>(d.n);
  p.k = static_cast<int32_t>(d.k);
  p.L = d.num_groups;
  p.n_out = static_cast<int32_t>(P->n_out);
  p.num_n_tiles = static_cast<int32_t>(ceil_div(d.n, P->bn));
  p.num_k_stages = static_cast<int32_t>(ceil_div(P->kbytes, bsgg::kBKBytes * P->slices));
  p.raster_w = P->bn == 256 ? 8 : 16;
  p.rn_b = static_cast<int32_t>(ceil_div(d.n, 128));
  p.kq_row = static_cast<int32_t>(ceil_div(ceil_div(P->n_out, P->sf_vec), 4));
  p.kq_col = static_cast<int32_t>(ceil_div(ceil_div(d.m_pad, P->sf_vec), 4));
  p.out_kind = d.out_format;
  p.sf_atoms = (!is_fp4_in(d.in_format) ? 1 : P->sf_vec == 32 ? 2 : 4) * P->slices;
  p.sf_v32 = P->sf_vec == 32 ? 1 : 0;
  p.want_col = d.want_col;
  p.gate_first = d.gate_first;
  p.tanh_s = d.tanh_clamp_s;
  p.tanh_rcp_s = d.tanh_clamp_s > 0.0f ? 1.0f / d.tanh_clamp_s : 0.0f;
  const double qmax = d.out_format == BSGG_OUT_E4M3 ? 448.0 : d.out_format == BSGG_OUT_E5M2 ? 57344.0 : 6.0;
  p.rcp_qmax = static_cast<float>(1.0 / qmax);
  p.idesc = make_idesc(d.in_format, P->bn, P->pair);
  p.bias = d.want_bias ? a->bias : nullptr;
  p.c_out = d.want_c ? a->c : nullptr;
  p.bias_kind = d.bias_format;
  p.c_kind = d.c_format;
  p.glu_kind = d.epilogue == BSGG_EPI_GEGLU ? 1 : 0;
  p.glu_limit = d.glu_limit;
  p.glu_gamma = d.glu_alpha == 0.0f ? 1.0f : d.glu_alpha;
  if (d.want_rht) {
    p.rht = a->rht;
    p.sfrht = static_cast<uint8_t*>(a->sfrht);
    p.rht_norm_const = a->rht_norm_const;
    p.rht_kind = d.rht_format == BSGG_OUT_E2M1 ? bsgg::OK_E2M1 : bsgg::OK_BF16;
    p.kq_rht = static_cast<int32_t>(ceil_div(ceil_div(P->n_out, 16), 4));
    p.rht_colwise = d.want_rht == 2 ? 1 : 0;
  }
  if (is_bwd_epi(d.epilogue)) {
    p.saved_c = a->saved_c;
    p.saved_c_kind = d.saved_c_format;
    p.beta = a->beta;
    p.dprob = a->dprob;
    p.bwd_kind = d.epilogue == BSGG_EPI_DGEGLU ? 1 : 0;
    p.dbias = a->dbias;
    p.situ_b1 = d.situ_beta1 == 0.0f ? 1.0f : d.situ_beta1;
    p.situ_b2 = d.situ_beta2 == 0.0f ? 1.0f : d.situ_beta2;
    const bool cust = d.dgeglu_custom != 0;
    p.geglu_a = cust ? d.dgeglu_alpha : 1.702f;
    p.clamp_min = cust ? d.dgeglu_clamp_min : -7.0f;
    p.clamp_max = cust ? d.dgeglu_clamp_max : 7.0f;
    p.lin_offset = cust ? d.dgeglu_linear_offset : 1.0f;
  }
  if (d.discrete_b) {
    p.b_maps = P->maps;
    p.maps_bad = reinterpret_cast<const uint32_t*>(P->maps + 2 * d.num_groups);
  }
  p.force_timeout = P->force_timeout ? 1u : 0u;
  // a test that makes the range checks fire also shortens the waits: the CTA
  // that stops loading leaves its partner's barriers incomplete
  p.wait_limit_ns = (P->force_timeout || P->dbg_margin) ? kTestWaitLimitNs : bsgg::kWaitLimitNs;
  p.dbg_rows = static_cast<int32_t>(d.m_pad - P->dbg_margin);

  // an upper bound of the scheduling units (pairs may add one 256-row tile
  // row per group)
  const bool cl = P->pair;
  const int64_t rows = cl ? ceil_div(d.m_pad, 256) + d.num_groups : d.m_pad / bsgg::kBM;
  const int64_t tiles = rows * p.num_n_tiles;
  L.grid = static_cast<int>(std::min<int64_t>(P->grid, cl ? 2 * tiles : tiles));
  L.pair = P->pair;
  L.bn = P->bn;
  L.epi = P->epi;
  L.outc = P->outc;
  L.stream = s;
  if (d.discrete_b) {
    const unsigned threads = static_cast<unsigned>(ceil_div(d.num_groups, 32) * 32);
    expert_maps_kernel<<<1, threads, 0, s>>>(L.tmB, L.tmSFB, a->b_ptrs, a->sfb_ptrs,
                                             d.in_format != BSGG_IN_BF16 ? 1 : 0, a->padded_offsets,
                                             d.num_groups, P->maps, P->status);
    if (cudaGetLastError() != cudaSuccess) return BSGG_ERR_CUDA;
  }
  cudaError_t e;
  if (is_bwd_epi(d.epilogue)) {
    if (d.in_format == BSGG_IN_BF16)
      e = P->pair ? bsgg::launch_bf16_pair_bwd(L)
          : P->bn == 256 ? bsgg::launch_bf16_256_bwd(L) : bsgg::launch_bf16_128_bwd(L);
    else if (is_f4e8_in(d.in_format))
      e = P->pair ? bsgg::launch_f4e8_pair_bwd(L)
          : P->bn == 256 ? bsgg::launch_f4e8_256_bwd(L) : bsgg::launch_f4e8_128_bwd(L);
    else if (d.in_format == BSGG_IN_NVFP4)
      e = P->pair ? bsgg::launch_nvf4_pair_bwd(L)
          : P->bn == 256 ? bsgg::launch_nvf4_256_bwd(L) : bsgg::launch_nvf4_128_bwd(L);
    else
      e = P->pair ? bsgg::launch_mxf8_pair_bwd(L)
          : P->bn == 256 ? bsgg::launch_mxf8_256_bwd(L) : bsgg::launch_mxf8_128_bwd(L);
  } else if (is_f4e8_in(d.in_format))
    e = P->pair ? bsgg::launch_f4e8_pair(L)
        : P->bn == 256 ? bsgg::launch_f4e8_256(L) : bsgg::launch_f4e8_128(L);
  else if (d.in_format == BSGG_IN_NVFP4)
    e = P->pair ? bsgg::launch_nvf4_pair(L)
        : P->bn == 256 ? bsgg::launch_nvf4_256(L) : bsgg::launch_nvf4_128(L);
  else
    e = P->pair ? bsgg::launch_mxf8_pair(L)
        : P->bn == 256 ? bsgg::launch_mxf8_256(L) : bsgg::launch_mxf8_128(L);
  return e == cudaSuccess ? BSGG_OK : BSGG_ERR_CUDA;
}

int32_t bsgg_launches_per_run(const bsgg_plan* P) {
  if (!P) return -1;
  return P->desc.discrete_b ? 2 : 1;   // the per-expert descriptor kernel, then the GEMM
}

bsgg_status bsgg_debug_force_timeout(bsgg_plan* P, int32_t enable) {
  if (!P || (enable != 0 && enable != 1)) return BSGG_ERR_INVALID_ARG;
  P->force_timeout = enable != 0;
  return BSGG_OK;
}

bsgg_status bsgg_query_device_status(bsgg_plan* P, void* stream) {
  if (!P) return BSGG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSGG_ERR_CUDA;
  uint32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpy(w, P->status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BSGG_ERR_CUDA;
  if (cudaMemset(P->status, 0, sizeof(w)) != cudaSuccess) return BSGG_ERR_CUDA;
  if (w[0] & bsgg::kStatusBounds) std::memcpy(P->violation, w + 1, sizeof(P->violation));
  return status_of_word(w[0]);
}

int32_t bsgg_debug_bounds_checked(void) { return bsgg::kDebugBounds ? 1 : 0; }

bsgg_status bsgg_debug_bounds_margin(bsgg_plan* P, int32_t rows) {
  if (!P || rows < 0 || rows % 128 != 0 || rows >= P->desc.m_pad) return BSGG_ERR_INVALID_ARG;
  if (!bsgg::kDebugBounds) return BSGG_ERR_UNSUPPORTED;
  P->dbg_margin = rows;
  return BSGG_OK;
}

bsgg_status bsgg_debug_bounds_violation(const bsgg_plan* P, uint32_t* site, uint32_t* value, uint32_t* limit) {
  if (!P || !site || !value || !limit) return BSGG_ERR_INVALID_ARG;
  *site = P->violation[0];
  *value = P->violation[1];
  *limit = P->violation[2];
  return BSGG_OK;
}

}  // extern "C"

namespace {

// bsgg_run_host / bsgg_run_host_async: the inputs present in `host` copied in,
// the kernel, the outputs present in `host` copied back, all on `stream`;
// `sync` waits for them.
bsgg_status run_host_impl(bsgg_plan* P, const bsgg_args* host, const bsgg_args* dev, void* stream,
                          uint64_t* h2d_bytes, uint64_t* d2h_bytes, bool sync) {
  if (!P || !host || !dev) return BSGG_ERR_INVALID_ARG;
  const bsgg_desc& d = P->desc;
  // discrete weights are taken as resident on the device
  if (d.discrete_b && (host->b || host->sfb || host->b_ptrs || host->sfb_ptrs)) return BSGG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t L = d.num_groups;
  const uint64_t sz_a = uint64_t(d.m_pad) * P->kbytes;
  const bool scaled = d.in_format != BSGG_IN_BF16;   // bfloat16 operands: no scale factors
  const uint64_t sz_sfa = scaled ? sf_bytes_impl(d.m_pad, d.k, P->sf_vec, 1) : 0;
  const uint64_t sz_b = uint64_t(L) * d.n * P->kbytes;
  const uint64_t sz_sfb = scaled ? sf_bytes_impl(d.n, d.k, P->sf_vec, L) : 0;
  const uint64_t sz_d = uint64_t(d.m_pad) * P->out_row_bytes;
  const uint64_t sz_sfd_row = sf_bytes_impl(d.m_pad, P->n_out, P->sf_vec, 1);
  const uint64_t sz_sfd_col = sf_bytes_impl(P->n_out, d.m_pad, P->sf_vec, 1);
  const bool bwd = is_bwd_epi(d.epilogue);
  const uint64_t sz_saved_c = bwd ? uint64_t(d.m_pad) * 2 * d.n * (d.saved_c_format == BSGG_OUT_F32 ? 4 : 2) : 0;
  const uint64_t n_amax = uint64_t(L) * (bwd ? 2 : 1);
  uint64_t in_bytes = 0, out_bytes = 0;
  auto h2d = [&](const void* h, const void* dv, uint64_t n) -> bool {
    if (!h) return true;
    if (!dv) return false;
    in_bytes += n;
    return cudaMemcpyAsync(const_cast<void*>(dv), h, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  auto d2h = [&](void* h, const void* dv, uint64_t n) -> bool {
    if (!h) return true;
    if (!dv) return false;
    out_bytes += n;
    return cudaMemcpyAsync(h, dv, n, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  };
  bool ok = h2d(host->a, dev->a, sz_a) && h2d(host->sfa, dev->sfa, sz_sfa) && h2d(host->b, dev->b, sz_b) &&
            h2d(host->sfb, dev->sfb, sz_sfb) &&
            h2d(host->padded_offsets, dev->padded_offsets, sizeof(int32_t) * L) &&
            h2d(host->alpha, dev->alpha, sizeof(float) * L) &&
            h2d(host->prob, dev->prob, sizeof(float) * d.m_pad) &&
            h2d(host->norm_const, dev->norm_const, sizeof(float)) &&
            h2d(d.want_bias ? host->bias : nullptr, dev->bias,
                uint64_t(L) * d.n * (d.bias_format == BSGG_OUT_F32 ? 4 : 2)) &&
            // backward: the saved C and beta in, dprob in (it is accumulated) and out
            h2d(bwd ? host->saved_c : nullptr, dev->saved_c, sz_saved_c) &&
            h2d(d.epilogue == BSGG_EPI_DSWIGLU || (!scaled && d.epilogue == BSGG_EPI_DGEGLU) ? host->beta : nullptr,
                dev->beta, sizeof(float) * L) &&
            h2d(bwd ? host->dprob : nullptr, dev->dprob, sizeof(float) * d.m_pad) &&
            h2d(d.want_rht ? host->rht_norm_const : nullptr, dev->rht_norm_const, sizeof(float)) &&
            h2d(bwd ? host->dbias : nullptr, dev->dbias, sizeof(float) * L * P->n_out);
  if (!ok) return BSGG_ERR_CUDA;
  bsgg_status st = bsgg_run(P, dev, stream);
  if (st != BSGG_OK) return st;
  ok = d2h(host->d, dev->d, sz_d) && d2h(host->d_col, dev->d_col, d.want_col ? sz_d : 0) &&
       d2h(host->sfd_row, dev->sfd_row, sz_sfd_row) &&
       d2h(host->sfd_col, dev->sfd_col, d.want_col ? sz_sfd_col : 0) &&
       d2h(host->amax, dev->amax, sizeof(float) * n_amax) &&
       d2h(bwd ? host->dprob : nullptr, dev->dprob, sizeof(float) * d.m_pad) &&
       d2h(bwd ? host->dbias : nullptr, dev->dbias, sizeof(float) * L * P->n_out) &&
       d2h(d.want_rht ? host->rht : nullptr, dev->rht,
           uint64_t(d.m_pad) * (d.rht_format == BSGG_OUT_E2M1 ? P->n_out / 2 : P->n_out * 2)) &&
       d2h(d.want_rht && d.rht_format == BSGG_OUT_E2M1 ? host->sfrht : nullptr, dev->sfrht,
           d.want_rht == 2 ? uint64_t(d.m_pad) * P->n_out / 16 : sf_bytes_impl(d.m_pad, P->n_out, 16, 1)) &&
       d2h(d.want_c ? host->c : nullptr, dev->c, uint64_t(d.m_pad) * d.n * out_elem_bits(d.c_format) / 8);
  if (!ok) return BSGG_ERR_CUDA;
  if (sync && cudaStreamSynchronize(s) != cudaSuccess) return BSGG_ERR_CUDA;
  if (h2d_bytes) *h2d_bytes = in_bytes;
  if (d2h_bytes) *d2h_bytes = out_bytes;
  return BSGG_OK;
}

}  // namespace

extern "C" {

bsgg_status bsgg_run_host(bsgg_plan* P, const bsgg_args* host, const bsgg_args* dev, void* stream,
                          uint64_t* h2d_bytes, uint64_t* d2h_bytes) {
  return run_host_impl(P, host, dev, stream, h2d_bytes, d2h_bytes, true);
}

bsgg_status bsgg_run_host_async(bsgg_plan* P, const bsgg_args* host, const bsgg_args* dev, void* stream,
                                uint64_t* h2d_bytes, uint64_t* d2h_bytes) {
  return run_host_impl(P, host, dev, stream, h2d_bytes, d2h_bytes, false);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.  For callers that cannot allocate device memory
// when they call in (a framework pool that already holds the device memory, a
// serving loop that must not let cudaMalloc/cudaFree synchronize the device, a
// plug-in whose host application owns memory): the status word that a plan
// would cudaMalloc lives instead in this file-scope device array, which every
// GPU that loads the library holds until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint32_t g_noalloc_scratch[BSGG_NOALLOC_SCRATCH_BYTES / sizeof(uint32_t)];

namespace {

constexpr size_t kNoAllocStatusBytes = 4 * sizeof(uint32_t);   // scratch one call needs: the status
                                                                 // word and the range-check record
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices];
int g_noalloc_sms[kNoAllocMaxDevices];
unsigned long long g_noalloc_ctx[kNoAllocMaxDevices];   // id of the context the address belongs to

// Unique id of the current context (driver cuCtxGetCurrent + cuCtxGetId,
// reached through the runtime's entry-point query), 0 if unavailable.  A
// context reset (cudaDeviceReset) gives the device a new context and a new id.
unsigned long long current_ctx_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Once per device (and again after that device's context was reset), with the
// device current: the array's device address (a host-side reference to the
// array is only a stand-in, never a device pointer) and the SM count.
bsgg_status noalloc_setup(int dev, uint32_t** scratch, int* sms) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  const unsigned long long ctx = current_ctx_id();
  if (!g_noalloc_addr[dev] || (ctx != 0 && ctx != g_noalloc_ctx[dev])) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return BSGG_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return BSGG_ERR_CUDA;
    g_noalloc_sms[dev] = n;
    g_noalloc_addr[dev] = addr;
    // the symbol lookup made the runtime's context current if it was not yet
    g_noalloc_ctx[dev] = ctx != 0 ? ctx : current_ctx_id();
  }
  *scratch = static_cast<uint32_t*>(g_noalloc_addr[dev]);
  *sms = g_noalloc_sms[dev];
  return BSGG_OK;
}

}  // namespace

extern "C" bsgg_status bsgg_run_noalloc(const bsgg_desc* desc, const bsgg_args* args, void* stream,
                                        int32_t wait_status) {
  const bsgg_status v = validate(desc);
  if (v != BSGG_OK) return v;
  // scratch this call needs: the status word, plus the per-expert tensor maps in
  // discrete weight mode (which never fit)
  const size_t need = kNoAllocStatusBytes + (desc->discrete_b ? maps_bytes(desc->num_groups) : 0);
  if (need > sizeof(g_noalloc_scratch)) return BSGG_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return BSGG_ERR_CUDA;
  uint32_t* scratch = nullptr;
  int sms = 0;
  const bsgg_status su = noalloc_setup(dev, &scratch, &sms);
  if (su != BSGG_OK) return su;

  // A plan on the stack, derived from `desc` exactly as bsgg_create derives
  // it, whose status word is the static scratch.
  bsgg_plan P{};
  if (init_plan(desc, dev, sms, &P) != BSGG_OK) return BSGG_ERR_CUDA;
  P.status = scratch;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, kNoAllocStatusBytes, s) != cudaSuccess) return BSGG_ERR_CUDA;
  const bsgg_status st = bsgg_run(&P, args, stream);
  if (st != BSGG_OK || !wait_status) return st;
  uint32_t w = 0;   // (the range-check record behind it is not reported here)
  if (cudaMemcpyAsync(&w, scratch, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return BSGG_ERR_CUDA;
  return status_of_word(w);
}
