// bsgg_kernel.cuh -- the persistent grouped block-scaled GEMM kernel for sm_103a.
//
// Tiles never straddle two expert groups because groups are padded to
// multiples of 128 rows ("Grouped GEMM + Quant (SM100)", Tiling and Cluster:
// tiles must not span groups).  Two cluster modes (CM) share this file:
//   * single (CM_SINGLE): one CTA computes a 128 x BN tile (BN = 128 or 256)
//     with tcgen05 .cta_group::1 MMAs.
//   * CTA pair (CM_PAIR, BN = 256): a cluster of two CTAs computes a
//     256 x 256 tile with .cta_group::2 MMAs: each CTA loads its own 128 rows
//     of A and half of the 256 rows of B, both CTAs hold all 256 columns' B
//     scales, the even CTA issues the MMAs and each CTA's tensor memory
//     receives its 128 rows of D.  Half the operand bytes per FLOP of 1-CTA
//     tiles.  A group with an odd number of 128-row tiles ends in a pair tile
//     whose odd half recomputes the even half's rows and stores nothing.
//     Every TMA load of a CTA writes only that CTA's own shared memory.
// Warp roles.  Eleven warps (352 threads) when the scale factors are copied:
//   warp 0      TMA producer: A, B[g] (128-byte swizzle) and the scale-factor
//               atoms (512-byte boxes) into a multi-stage ring; in a pair both
//               producers complete the even CTA's "full" barrier
//   warp 1      tensor-memory allocator and (even CTA) MMA issuer: block-scaled
//               tcgen05.mma (MXFP8 kind::mxf8f6f4 or NVFP4 kind::mxf4nvf4)
//   warp 10     (even CTA) scale copier: tcgen05.cp of each stage's scale atoms
//               to tensor memory, then a commit that releases the stage to the
//               MMA issuer.  A copy in the MMA thread's own tcgen05 queue stalls
//               the MMAs issued around it, so copies run from this thread.
//   warps 2..9  epilogue, two warps per 32-lane tensor-memory quadrant, each
//               owning half of the tile's columns: tcgen05.ld of the whole
//               half into registers (then the accumulator is released), alpha,
//               the activation and prob (Step 2), per-group amax or the row /
//               column block quantization (Step 3); D and D_col through a
//               shared-memory staging slot per warp and TMA stores (MXFP8 and
//               bfloat16 inputs) or direct vector stores
// FP4 inputs (sixteen warps, 512 threads) store the scales instead: the copies of an NVFP4 stage's twelve atoms held the
// tensor pipe back.  Warps 0 and 1 as above; warps 2..5 write the scales with
// tcgen05.st, one per lane quadrant, A's atoms without the copy path's
// four-fold replication (in a pair each CTA's warps write its own tensor
// memory and report to the even CTA); warps 6, 7 idle; warps 8..15 the
// epilogue.  Warps 0..7 give registers to the epilogue (setmaxnreg: 64 / 192).
// All waits are bounded; a wait that runs out raises a CTA-wide abort flag and
// a device status bit, and every role then drains its in-flight asynchronous
// work (again with a bound) and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace bsgg {

// Epilogue instances; EPI_SWIGLU also computes GeGLU (Params::glu_kind);
// EPI_DSWIGLU is the dSwiGLU backward, and the dGeGLU backward (Params::bwd_kind);
// EPI_DSITUGLU the dSiTU-GLU backward (its tanh and sech^2 need registers the
// other two instances must not give up).
enum : int { EPI_GATE = 0, EPI_SWIGLU = 1, EPI_SRELU = 2, EPI_DSWIGLU = 3, EPI_DSITUGLU = 4 };
__host__ __device__ constexpr bool is_bwd_inst(int epi) { return epi == EPI_DSWIGLU || epi == EPI_DSITUGLU; }
// Input class (template): MXFP8 (E4M3/E5M2 data, UE8M0 scales per 32), NVFP4
// (E2M1 data, E4M3 scales per 16), or E2M1 data with UE8M0 scales, whose block
// length (16 or 32) is a runtime choice (Params::sf_v32).  NVFP4 keeps its own
// instances: the runtime choices cost it 2 % on GB300.  IC_BF16: bfloat16 A
// and B without scale factors (the BF16 backend of the dGLU backward).
enum : int { IC_MXF8 = 0, IC_NVF4 = 1, IC_F4E8 = 2, IC_BF16 = 3 };
__host__ __device__ constexpr bool ic_fp4(int ic) { return ic == IC_NVF4 || ic == IC_F4E8; }
__host__ __device__ constexpr bool ic_scaled(int ic) { return ic != IC_BF16; }
// Output class (template) and exact output kind (runtime) of D.
enum : int { OUTC_FLOAT = 0, OUTC_FP8 = 1, OUTC_FP4 = 2 };
enum : int { OK_BF16 = 0, OK_F16 = 1, OK_F32 = 2, OK_E4M3 = 3, OK_E5M2 = 4, OK_E2M1 = 5 };

constexpr int kBM = 128;          // rows per CTA tile (TMEM lanes)
constexpr int kBKBytes = 128;     // K bytes per slice: one 128-byte swizzle span, one TMA box row
constexpr int kEpiWarps = 8;      // two warps per tensor-memory lane quadrant
constexpr int kStoreSlot = 2048;  // an epilogue warp's TMA-store staging bytes (32 rows of a D chunk and of D_col)
enum : int { CM_SINGLE = 0, CM_PAIR = 1 };
// K slices per pipeline stage (each slice one 128-byte box per operand and
// four MMAs).  Every instance takes one: two slices per stage (eight MMAs per
// barrier round trip, three stages in the shared memory of six) measured no
// faster on GB300 for the MXFP8 CTA pairs (FC1 +1 %, FC2 -4 %, skewed +0 %),
// so the ring stays deep rather than wide.
__host__ __device__ constexpr int stage_slices(int, int) { return 1; }
// Scale factors reach tensor memory by tcgen05.st from four warps (one per
// lane quadrant) for FP4 inputs, by tcgen05.cp from one thread otherwise (see
// the kernel's role table).  Measured on GB300: stores raise NVFP4 by 19 %
// (single) and 14 % (pairs) and lower MXFP8 pairs by 17 %.
template <bool FP4>
constexpr bool scale_stores() { return FP4; }
template <bool ST>
struct Roles {
  static constexpr int kThreads = ST ? 512 : 96 + 32 * kEpiWarps;
  static constexpr int kEpiFirst = ST ? 8 : 2;   // epilogue warps [kEpiFirst, kEpiFirst + 8)
  static constexpr int kCopyWarp = 10;           // tcgen05.cp mode: the copying warp
  // tcgen05.st mode: warps 0-7 drop to kLowRegs, warps 8-15 rise to kHighRegs;
  // 256 x kLowRegs + 256 x kHighRegs = 512 x 128, the launch's registers
  static constexpr int kLaunchRegs = 128;
  static constexpr int kLowRegs = 64;
  static constexpr int kHighRegs = 192;
};
static_assert(256 * Roles<true>::kLowRegs + 256 * Roles<true>::kHighRegs == 512 * Roles<true>::kLaunchRegs,
              "the register split must add up to the launch's registers");
constexpr int kMaxGroups = 1024;
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadOffsets = 2u;
constexpr uint32_t kStatusBadPointers = 4u;
constexpr uint32_t kStatusBounds = 8u;               // range-checking build: an index failed its check
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s per wait (Params::wait_limit_ns)
constexpr uint64_t kDrainLimitNs = 200000000ull;     // 0.2 s per drain wait

struct Params {
  const int32_t* offsets;
  const float* alpha;
  const float* prob;
  const float* norm_const;
  void* d;
  void* d_col;
  uint8_t* sfd_row;
  uint8_t* sfd_col;
  float* amax;
  uint32_t* status;
  int32_t m_pad, n, k, L;
  int32_t n_out;            // columns of D
  int32_t num_n_tiles;      // ceil(N / BN)
  int32_t num_k_stages;
  int32_t raster_w;         // n-tiles per raster band inside a group
  int32_t rn_b;             // 128-row SF row-blocks of one expert's B: ceil(N/128)
  int32_t kq_row;           // SF atoms per 128 rows of SFD_row: ceil(ceil(n_out/v)/4)
  int32_t kq_col;           // SF atoms per 128 columns of SFD_col: ceil(ceil(m_pad/v)/4)
  int32_t out_kind;         // OK_*
  // IC_F4E8 instances: scale atoms a stage loads (4: one scale per 16 values;
  // 2: one per 32, each written into both 16-value slots it covers) and the
  // block length of the input (and so of the quantized outputs)
  int32_t sf_atoms;
  int32_t sf_v32;           // 1: blocks of 32 values, 0: of 16
  int32_t want_col;
  int32_t gate_first;
  float tanh_s, tanh_rcp_s; // soft clamp s and 1/s (s = 0: off)
  float rcp_qmax;           // fp32(1/q_max) of the output format
  uint32_t idesc;           // tcgen05 instruction descriptor without scale ids
  uint32_t force_timeout;   // test of the failure path: the MMA thread first waits on a
                            // barrier nothing completes, so every role gives up and returns
  uint64_t wait_limit_ns;   // bound of every barrier wait (kWaitLimitNs; shorter in that test)
  int32_t dbg_rows;         // range-checking build: rows of A, D, prob the checks accept (m_pad,
                            // less a margin a test may set to see the checks fire)
  // "Grouped GEMM + GLU + Hadamard + Quant (SM100)", Equations: C = alpha_g * acc +
  // bias_g[n], optionally stored before any clamp or activation; GLU clamp and scale
  const void* bias;         // (L, N), N contiguous, or null
  void* c_out;              // (m_pad, N) N-major, or null
  int32_t bias_kind;        // OK_BF16, OK_F16 or OK_F32
  int32_t c_kind;           // OK_BF16 or OK_F16; with MXFP8 inputs also OK_F32, OK_E4M3, OK_E5M2, OK_E2M1
  int32_t glu_kind;         // EPI_SWIGLU instances: 0 = SwiGLU, 1 = GeGLU
  float glu_limit;          // both GLU halves clamped to [-glu_limit, glu_limit]; 0 = none
  float glu_gamma;          // GLU output scale (1 = none)
  // dSwiGLU backward ("Grouped GEMM + dGLU (SM100)"): the saved forward C
  // (m_pad, 2N), its per-group scale, and the accumulated dprob (m_pad)
  const void* saved_c;
  int32_t saved_c_kind;     // OK_BF16, OK_F16 or OK_F32
  const float* beta;        // dSwiGLU only
  float* dprob;
  int32_t bwd_kind;         // EPI_DSWIGLU instances: 0 = dSwiGLU, 1 = dGeGLU
  float* dbias;             // backward: (L, n_out) accumulated row sums of D per group, or null
  float geglu_a, clamp_min, clamp_max, lin_offset;   // dGeGLU
  float situ_b1, situ_b2;                            // dSiTU-GLU
  // rowwise Hadamard output of bf16-rounded D ("Grouped GEMM + GLU + Hadamard +
  // Quant (SM100)"): bf16 or NVFP4 with E4M3 scales per 16 (SFRHT)
  void* rht;                // (m_pad, n_out), or null
  uint8_t* sfrht;
  const float* rht_norm_const;
  int32_t rht_kind;         // OK_BF16 or OK_E2M1
  int32_t kq_rht;           // SF atoms per 128 rows of SFRHT: ceil(ceil(n_out/16)/4)
  int32_t rht_colwise;      // 1: 16-token blocks per column, per-expert transposed (NVFP4)
  // discrete weight mode: per-expert tensor maps {B_g, SFB_g} (2 per expert, in
  // global memory) and the flag their writer raises for a bad pointer; null in
  // dense mode
  const CUtensorMap* b_maps;
  const uint32_t* maps_bad;
};

// SCALED = false (bfloat16 operands): no scale buffers, 64 K elements per
// 128-byte stage, 16 per MMA.
template <bool FP4, int BN, bool PAIR, bool SCALED = true, int SL = 1>
struct Layout {
  static_assert(BN == 128 || BN == 256, "tile width");
  static_assert(!PAIR || BN == 256, "CTA pairs use 256 x 256 tiles");
  static_assert(SL == 1 || SL == 2, "one or two K slices per stage");
  static constexpr int kSlices = SL;
  static constexpr int kStageK = SL * kBKBytes;            // K bytes per stage
  static constexpr int kHalves = BN / 128;                 // 128-row SF blocks of the MMA's N
  static constexpr int kBRows = PAIR ? BN / 2 : BN;        // B rows held by this CTA
  static constexpr int kAtoms = (!SCALED ? 0 : FP4 ? 4 : 1) * SL;        // SF atoms per stage per 128 rows
  static constexpr int kKElems = (!SCALED ? 64 : FP4 ? 256 : 128) * SL;  // K elements per stage
  static constexpr int kMmaK = !SCALED ? 16 : FP4 ? 64 : 32;             // K elements per MMA instruction
  static constexpr int kMmas = 4 * SL;                                   // MMAs per stage
  static constexpr int kASlice = kBM * kBKBytes;           // one slice of A (a 128-byte swizzled box)
  static constexpr int kBSlice = kBRows * kBKBytes;
  static constexpr int kABytes = kASlice * SL;
  static constexpr int kBBytes = kBSlice * SL;
  static constexpr int kSfaBytes = kAtoms * 512;
  static constexpr int kSfbBytes = kAtoms * kHalves * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;   // one CTA's bytes
  static constexpr int kStages = (221184 / kStageBytes) > 8 ? 8 : (221184 / kStageBytes);
  // two accumulators where they fit beside the scale slots: 128-column tiles,
  // and 256-column tiles without scales (bfloat16 operands)
  static constexpr int kNumAcc = (BN == 128 || !SCALED) ? 2 : 1;
  static constexpr int kSfaCols = kAtoms * 4;
  static constexpr int kSfbCols = kAtoms * kHalves * 4;
  static constexpr int kSfColsPerStage = kSfaCols + kSfbCols;
  static constexpr int kTmemCols = 512;
  static_assert(kNumAcc * BN + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
  // shared-memory map, relative to a 1024-byte aligned base
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr int kOffBars = kOffSfb + kStages * kSfbBytes;
  static constexpr int kNumBars = 4 * kStages + 2 * kNumAcc + 2;
  static constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemHolder + 4;
  static constexpr int kOffTrows = kOffAbort + 12;
  static constexpr int kOffOffsets = kOffTrows + 4 * kMaxGroups;
  // the epilogue warps' TMA-store staging slots, where they fit beside the ring
  static constexpr int kOffStore = (kOffOffsets + 4 * kMaxGroups + 127) / 128 * 128;
  static constexpr int kStoreBytes = kEpiWarps * kStoreSlot;
  static constexpr bool kTmaStore = kOffStore + kStoreBytes + 1024 <= 232448;
  static constexpr int kSmemBytes = (kTmaStore ? kOffStore + kStoreBytes : kOffOffsets + 4 * kMaxGroups) +
                                    1024;   // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffSfa % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

// Range-checking build (compiled with BSGG_DEBUG_BOUNDS): every TMA box
// origin, scale-factor offset and output index is checked against the
// problem's extents before use.  A failed check records the first failure
// (site, value, limit in status words 1..3), raises kStatusBounds and skips the
// access; in the producer it also raises the CTA's abort flag, so that every
// role drains and returns as after a timeout.  Without the macro the checks
// compile to nothing.
#ifdef BSGG_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif
// check sites (status word 1)
enum : uint32_t {
  kSiteARows = 1, kSiteBRow = 2, kSiteBSlice = 3, kSiteSfa = 4, kSiteSfb = 5, kSiteK = 6,
  kSiteDRow = 10, kSiteDCol = 11, kSiteSfdRow = 12, kSiteSfdCol = 13, kSiteAmax = 14, kSiteC = 15,
  kSiteRht = 16, kSiteDprob = 17, kSiteDbias = 18, kSiteGroup = 19
};
static __device__ __noinline__ void bounds_fail(uint32_t* status, uint32_t site, int64_t v, int64_t lim) {
  if (atomicCAS(status + 1, 0u, site) == 0u) {
    status[2] = static_cast<uint32_t>(v);
    status[3] = static_cast<uint32_t>(lim);
  }
  atomicOr(status, kStatusBounds);
}
// 0 <= v < lim (always true without BSGG_DEBUG_BOUNDS).
__device__ __forceinline__ bool in_range(uint32_t* status, uint32_t site, int64_t v, int64_t lim) {
  if constexpr (!kDebugBounds) {
    return true;
  } else {
    if (v >= 0 && v < lim) return true;
    bounds_fail(status, site, v, lim);
    return false;
  }
}

// Byte offset of the scale of (row, k-block) in a swizzled SF buffer whose
// rows hold kq 512-byte atoms: 128-row block, then k-atom, then inside the atom
// 16 bytes per row-in-32, 4 bytes per 32-row quarter, 1 byte per k-block.
__device__ __forceinline__ int64_t sf_off(int64_t row, int64_t kblk, int64_t kq) {
  return ((row >> 7) * kq + (kblk >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kblk & 3);
}

// Scheduling units of a group with mt 128-row tiles: tiles (single) or
// 256-row tile rows (pair).
template <int CM>
__device__ __forceinline__ int group_units(int mt) {
  return CM == CM_PAIR ? (mt + 1) / 2 : mt;
}

// Tile t of the static schedule -> (group, this CTA's 128-row tile, n-tile).
// A "tile row" is 128 rows (1-CTA) or 256 rows (pair); group g holds
// trows_g = ceil(m-tiles_g / (PAIR ? 2 : 1)) of them and s_trow is their
// inclusive prefix sum.  Tiles of group g occupy [ntn * trow_start, ntn *
// trow_end); inside a group the n-tiles are walked in bands of raster_w, every
// tile row of the group before the next band, so that a band of B stays in L2
// while the group's rows pass over it.  Empty groups own no tiles.  `valid` is
// false only for the odd half of a pair tile past the group's last row; that
// half then reuses the even half's rows (m_load) and stores nothing.
template <int CM>
__device__ __forceinline__ void decode_tile(int t, const Params& p, const int32_t* s_off, const int32_t* s_trow,
                                            uint32_t rank, int& g, int& m_load, int& n_tile, bool& valid) {
  constexpr bool PAIR = CM == CM_PAIR;
  const int ntn = p.num_n_tiles;
  const int u = t / ntn;
  int lo = 0, hi = p.L;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_trow[mid] > u) hi = mid; else lo = mid + 1;
  }
  g = lo;
  const int tr0 = g ? s_trow[g - 1] : 0;
  const int trg = s_trow[g] - tr0;
  const int r = t - tr0 * ntn;
  const int W = p.raster_w;
  const int band = r / (trg * W);
  const int w = min(W, ntn - band * W);
  const int rr = r - band * trg * W;
  const int lt = rr / w;
  n_tile = band * W + rr % w;
  const int m0 = (g ? s_off[g - 1] : 0) / kBM;
  if (PAIR) {
    const int m = m0 + 2 * lt + static_cast<int>(rank);
    valid = m < s_off[g] / kBM;
    m_load = valid ? m : m - 1;
  } else {
    m_load = m0 + lt;
    valid = true;
  }
}

// UE8M0 code of the smallest power of two >= sf (sf >= 0); 0 for sf = 0.
__device__ __forceinline__ uint32_t ue8m0_ceil(float sf) {
  if (sf != sf) return 0xFFu;
  const uint32_t b = __float_as_uint(sf);
  const uint32_t e = b >> 23, m = b & 0x7FFFFFu;
  uint32_t code;
  if (e == 0) code = (m > 0x400000u) ? 1u : 0u;   // subnormal: above 2^-127 rounds to 2^-126
  else code = e + (m != 0u ? 1u : 0u);
  return code > 254u ? 254u : code;
}
// 2^(127 - code) as a float (exact; code 254 gives the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_recip(uint32_t code) {
  return code < 254u ? __uint_as_float((254u - code) << 23) : __uint_as_float(0x00400000u);
}

// Step 3 block scale: SFD = norm * amax * (1/q_max), encoded in the input's
// scale format; returns the code and the factor norm / decode(SFD) (0 for an
// all-zero block).
template <bool E4M3_SCALE>
__device__ __forceinline__ void block_scale(float am, float norm, float rcp_qmax, uint32_t& code,
                                            float& scale) {
  const float sf = (norm * am) * rcp_qmax;
  if (E4M3_SCALE) {
    code = cvt_e4m3x2(sf, 0.0f) & 0xFFu;
    const float sfd = e4m3_to_float(code);
    scale = (am == 0.0f || sfd == 0.0f) ? 0.0f : __fdiv_rn(norm, sfd);
  } else {
    code = ue8m0_ceil(sf);
    scale = (am == 0.0f) ? 0.0f : norm * ue8m0_recip(code);
  }
}

__device__ __forceinline__ void st_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// 16 bytes of a row's output chunk, to global memory (a pointer) or, for TMA
// stores, to a shared-memory staging address (a 32-bit shared address).
__device__ __forceinline__ void put16(uint8_t* g, int off, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  st_v4(g + off, a, b, c, d);
}
__device__ __forceinline__ void put16(uint32_t s, int off, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  st_shared_v4(s + off, a, b, c, d);
}

__device__ __forceinline__ float as_f32(float x) { return x; }
__device__ __forceinline__ float as_f32(uint32_t x) { return __uint_as_float(x); }

// 32 values of one row (floats, or fp32 bit patterns) stored as bf16 or f16
// at `dst` (64 bytes, 16-byte aligned).
template <typename Dst, typename T>
__device__ __forceinline__ void store_h32_to(Dst dst, const T* v, int kind) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (kind == OK_BF16) {
      __nv_bfloat162 h = __floats2bfloat162_rn(as_f32(v[2 * i]), as_f32(v[2 * i + 1]));
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __half2 h = __floats2half2_rn(as_f32(v[2 * i]), as_f32(v[2 * i + 1]));
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) put16(dst, 16 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}
template <typename T>
__device__ __forceinline__ void store_h32(void* dst, const T* v, int kind) {
  store_h32_to(static_cast<uint8_t*>(dst), v, kind);
}

// Adds the 32 bias values at `src` (bf16, f16 or f32; 16-byte aligned) to 32
// fp32 bit patterns in place.  Every lane of the warp reads the same addresses.
__device__ __forceinline__ void add_bias32(uint32_t* v, const void* src, int kind) {
  auto add = [&](int i, float b) { v[i] = __float_as_uint(__uint_as_float(v[i]) + b); };
  if (kind == OK_F32) {
    const float4* b = static_cast<const float4*>(src);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = __ldg(b + i);
      add(4 * i, x.x); add(4 * i + 1, x.y); add(4 * i + 2, x.z); add(4 * i + 3, x.w);
    }
  } else {
    const uint4* b = static_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = __ldg(b + i);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (kind == OK_BF16) {
          add(8 * i + 2 * j, __uint_as_float(w[j] << 16));
          add(8 * i + 2 * j + 1, __uint_as_float(w[j] & 0xFFFF0000u));
        } else {
          const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
          add(8 * i + 2 * j, __low2float(h));
          add(8 * i + 2 * j + 1, __high2float(h));
        }
      }
    }
  }
}

// 32 consecutive values (bf16, f16 or f32; 16-byte aligned) read as floats.
__device__ __forceinline__ void load_f32x32(float (&v)[32], const void* src, int kind) {
  if (kind == OK_F32) {
    const float4* b = static_cast<const float4*>(src);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = __ldg(b + i);
      v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
    }
  } else {
    const uint4* b = static_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = __ldg(b + i);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (kind == OK_BF16) {
          v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
          v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        } else {
          const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
          v[8 * i + 2 * j] = __low2float(h);
          v[8 * i + 2 * j + 1] = __high2float(h);
        }
      }
    }
  }
}

// Two products: one packed f32x2 multiply, or (PACKED false: the 256-column
// backward epilogues, whose register allocation spills with the packed form)
// two scalar ones; the same round-to-nearest results either way.
template <bool PACKED>
__device__ __forceinline__ float2 mul_pair(float a0, float a1, float b0, float b1) {
  if (PACKED) return __fmul2_rn(make_float2(a0, a1), make_float2(b0, b1));
  return make_float2(a0 * b0, a1 * b1);
}

// 32 values of one row -> quantized codes stored at `dst` (32 bytes for FP8,
// 16 bytes for FP4), each value multiplied by its block's scale first.
template <int OUTC, bool PACKED = true, typename Dst>
__device__ __forceinline__ void store_q32_to(Dst dst, const float (&v)[32], const float (&sc)[32], int out_kind) {
  if (OUTC == OUTC_FP8) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t lo, hi;
      const float2 a = mul_pair<PACKED>(v[4 * i], v[4 * i + 1], sc[4 * i], sc[4 * i + 1]);
      const float2 b = mul_pair<PACKED>(v[4 * i + 2], v[4 * i + 3], sc[4 * i + 2], sc[4 * i + 3]);
      if (out_kind == OK_E4M3) {
        lo = cvt_e4m3x2(a.x, a.y);
        hi = cvt_e4m3x2(b.x, b.y);
      } else {
        lo = cvt_e5m2x2(a.x, a.y);
        hi = cvt_e5m2x2(b.x, b.y);
      }
      w[i] = lo | (hi << 16);
    }
    put16(dst, 0, w[0], w[1], w[2], w[3]);
    put16(dst, 16, w[4], w[5], w[6], w[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 8 * i + 2 * j;
        const float2 q = mul_pair<PACKED>(v[e], v[e + 1], sc[e], sc[e + 1]);
        x |= cvt_e2m1x2(q.x, q.y) << (8 * j);
      }
      w[i] = x;
    }
    put16(dst, 0, w[0], w[1], w[2], w[3]);
  }
}
template <int OUTC, bool PACKED = true>
__device__ __forceinline__ void store_q32(void* dst, const float (&v)[32], const float (&sc)[32], int out_kind) {
  store_q32_to<OUTC, PACKED>(static_cast<uint8_t*>(dst), v, sc, out_kind);
}

// The codes of 32 values of one row whose column j is scaled by lane j's
// `scale` (the 32-row column blocks of the MXFP8 path), each factor fetched
// from its lane as its codes are formed.
template <int OUTC, typename Dst>
__device__ __forceinline__ void store_q32_cols_to(Dst dst, const float (&v)[32], float scale, int out_kind) {
  auto scaled = [&](int e) {
    return __fmul2_rn(make_float2(v[e], v[e + 1]),
                      make_float2(__shfl_sync(0xffffffffu, scale, e), __shfl_sync(0xffffffffu, scale, e + 1)));
  };
  if (OUTC == OUTC_FP8) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 a = scaled(4 * i), b = scaled(4 * i + 2);
      const uint32_t lo = out_kind == OK_E4M3 ? cvt_e4m3x2(a.x, a.y) : cvt_e5m2x2(a.x, a.y);
      const uint32_t hi = out_kind == OK_E4M3 ? cvt_e4m3x2(b.x, b.y) : cvt_e5m2x2(b.x, b.y);
      w[i] = lo | (hi << 16);
    }
    put16(dst, 0, w[0], w[1], w[2], w[3]);
    put16(dst, 16, w[4], w[5], w[6], w[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 q = scaled(8 * i + 2 * j);
        x |= cvt_e2m1x2(q.x, q.y) << (8 * j);
      }
      w[i] = x;
    }
    put16(dst, 0, w[0], w[1], w[2], w[3]);
  }
}

// The stored pre-activation C of one row's 32-column chunk (fp32 bit patterns):
// bf16 / f16 inline; f32, or, without a scale factor, the saturating
// round-to-nearest FP8 / FP4 conversion of C itself, in a function of its own
// (called only for those formats, so that the bias / C instances keep their
// registers for the common bf16 / f16 C).
struct C32 {
  uint32_t v[32];
};
static __device__ __noinline__ void store_c32_wide(void* c_out, int64_t rc, int kind, C32 c) {
  if (kind == OK_F32) {
    uint32_t* dst = static_cast<uint32_t*>(c_out) + rc;
#pragma unroll
    for (int i = 0; i < 8; ++i) st_v4(dst + 4 * i, c.v[4 * i], c.v[4 * i + 1], c.v[4 * i + 2], c.v[4 * i + 3]);
  } else if (kind == OK_E2M1) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        x |= cvt_e2m1x2(__uint_as_float(c.v[8 * i + 2 * j]), __uint_as_float(c.v[8 * i + 2 * j + 1])) << (8 * j);
      w[i] = x;
    }
    st_v4(static_cast<uint8_t*>(c_out) + rc / 2, w[0], w[1], w[2], w[3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float a = __uint_as_float(c.v[4 * i]), b = __uint_as_float(c.v[4 * i + 1]);
      const float d = __uint_as_float(c.v[4 * i + 2]), e = __uint_as_float(c.v[4 * i + 3]);
      const uint32_t lo = kind == OK_E4M3 ? cvt_e4m3x2(a, b) : cvt_e5m2x2(a, b);
      const uint32_t hi = kind == OK_E4M3 ? cvt_e4m3x2(d, e) : cvt_e5m2x2(d, e);
      w[i] = lo | (hi << 16);
    }
    uint8_t* dst = static_cast<uint8_t*>(c_out) + rc;
    st_v4(dst, w[0], w[1], w[2], w[3]);
    st_v4(dst + 16, w[4], w[5], w[6], w[7]);
  }
}
__device__ __forceinline__ void store_c32(const Params& p, const uint32_t* v, int row, int col0) {
  const int64_t rc = static_cast<int64_t>(row) * p.n + col0;   // element offset
  if (p.c_kind == OK_BF16 || p.c_kind == OK_F16) {
    store_h32(static_cast<uint16_t*>(p.c_out) + rc, v, p.c_kind);
  } else {
    C32 c;
#pragma unroll
    for (int i = 0; i < 32; ++i) c.v[i] = v[i];
    store_c32_wide(p.c_out, rc, p.c_kind, c);
  }
}

// TMA-store staging of one epilogue warp: a kStoreSlot-byte shared-memory slot
// (0: the warp stores its chunks directly) that holds the warp's 32 rows of a
// D chunk, and with column outputs the D_col chunk half a slot after it, and
// the tensor maps they are stored through.
struct OutStage {
  uint32_t slot;
  const CUtensorMap* d;
  const CUtensorMap* d_col;
};

// Step 3 (or the 16/32-bit store) of one 32-column chunk of D of one row:
// v[32] at D columns [col0, col0 + 32).  Row blocks of v columns lie inside the
// chunk; column blocks of v rows span the warp's 32 lanes (its 32 rows).  With
// a staging slot the warp writes its 32 rows' chunk bytes into it (row after
// row, as the TMA box lays them out) and one lane stores the whole 32-row box
// with a TMA store; the scale factors are stored directly either way.
template <int IC, int OUTC, bool SCALAR = false>
__device__ __forceinline__ void output_chunk(const Params& p, const float (&v)[32], int row, int col0,
                                             float norm, int lane, int kblk_col, float& amax_local,
                                             const OutStage& os) {
  if constexpr (kDebugBounds) {
    // the chunk's D / D_col bytes and the scale-factor bytes it writes; the
    // whole warp skips the chunk when a lane fails (the column blocks are
    // warp-collective)
    bool ok = in_range(p.status, kSiteDRow, row, p.dbg_rows) && in_range(p.status, kSiteDCol, col0 + 31, p.n_out);
    if (OUTC != OUTC_FLOAT) {
      const bool v16 = ic_fp4(IC) && !(IC == IC_F4E8 && p.sf_v32);
      const int kr = v16 ? col0 / 16 + 1 : col0 / 32;                    // last row block written
      const int64_t row_bytes = 512 * static_cast<int64_t>((p.m_pad + 127) / 128) * p.kq_row;
      ok = ok && in_range(p.status, kSiteSfdRow, kr >> 2, p.kq_row) &&
           in_range(p.status, kSiteSfdRow, sf_off(row, kr, p.kq_row), row_bytes);
      if (p.want_col) {
        const int kc = v16 ? 2 * kblk_col + 1 : kblk_col;                  // last column block written
        const int64_t col_bytes = 512 * static_cast<int64_t>((p.n_out + 127) / 128) * p.kq_col;
        ok = ok && in_range(p.status, kSiteSfdCol, kc >> 2, p.kq_col) &&
             in_range(p.status, kSiteSfdCol, sf_off(col0 + 31, kc, p.kq_col), col_bytes);
      }
    }
    if (__any_sync(0xffffffffu, !ok)) return;
  }
  // bytes of one row's chunk: 16-bit floats, FP8 codes, packed FP4 codes
  constexpr int kChunkBytes = OUTC == OUTC_FLOAT ? 64 : OUTC == OUTC_FP8 ? 32 : 16;
  // (FP4 inputs store directly: their 128-register instances spill with the
  // staging path, measured 1 % slower on the NVFP4 workload)
  const bool staged = !ic_fp4(IC) && os.slot != 0u && !(OUTC == OUTC_FLOAT && p.out_kind == OK_F32);
  if (staged) {
    // the slot's previous chunk has been read by its TMA store
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }
  const uint32_t d_stage = os.slot + static_cast<uint32_t>(lane * kChunkBytes);
  const uint32_t dcol_stage = os.slot + static_cast<uint32_t>(kStoreSlot / 2 + lane * kChunkBytes);
  int store_x = 0;                                   // the chunk's first byte within a row
  if (OUTC == OUTC_FLOAT) {
#pragma unroll
    for (int i = 0; i < 32; ++i) amax_local = fmaxf(amax_local, fabsf(v[i]));
    store_x = 2 * col0;
    if (p.out_kind == OK_F32) {
      float* dst = static_cast<float*>(p.d) + static_cast<int64_t>(row) * p.n_out + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        st_v4(dst + 4 * i, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
              __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
    } else if (staged) {
      store_h32_to(d_stage, &v[0], p.out_kind);
    } else {
      store_h32(static_cast<uint16_t*>(p.d) + static_cast<int64_t>(row) * p.n_out + col0, &v[0], p.out_kind);
    }
  } else {
    // ---- row blocks in the input's scale type and block length: 32 with UE8M0
    // scales for MXFP8; for FP4 two 16-value blocks with E4M3 or UE8M0 scales,
    // which one scale per 32 values (MXFP4) joins into one block
    constexpr bool FP4 = ic_fp4(IC);
    constexpr bool e4m3_sf = IC == IC_NVF4;
    const bool v32 = IC == IC_F4E8 && p.sf_v32;
    const int64_t row_bytes = (OUTC == OUTC_FP8) ? p.n_out : p.n_out / 2;
    const int64_t col_byte0 = (OUTC == OUTC_FP8) ? col0 : col0 / 2;
    float sc[32];
    if (FP4) {
      float am[2];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        am[b] = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am[b] = fmaxf(am[b], fabsf(v[b * 16 + i]));
      }
      if (v32) am[0] = am[1] = fmaxf(am[0], am[1]);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint32_t code;
        float s;
        if (e4m3_sf) block_scale<true>(am[b], norm, p.rcp_qmax, code, s);
        else block_scale<false>(am[b], norm, p.rcp_qmax, code, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) sc[b * 16 + i] = s;
        if (!v32) p.sfd_row[sf_off(row, col0 / 16 + b, p.kq_row)] = static_cast<uint8_t>(code);
        else if (b == 0) p.sfd_row[sf_off(row, col0 / 32, p.kq_row)] = static_cast<uint8_t>(code);
      }
    } else {
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
      uint32_t code;
      float s;
      block_scale<false>(am, norm, p.rcp_qmax, code, s);
#pragma unroll
      for (int i = 0; i < 32; ++i) sc[i] = s;
      p.sfd_row[sf_off(row, col0 / 32, p.kq_row)] = static_cast<uint8_t>(code);
    }
    store_x = static_cast<int>(col_byte0);
    if (staged) store_q32_to<OUTC, !SCALAR>(d_stage, v, sc, p.out_kind);
    else store_q32<OUTC, !SCALAR>(static_cast<uint8_t*>(p.d) + row * row_bytes + col_byte0, v, sc, p.out_kind);
    // ---- column blocks of v rows: the warp's 32 lanes are its 32 rows
    if (p.want_col) {
      if (!FP4) {
        // v = 32: column j's max over the warp's rows; lane j keeps it,
        // encodes that column's scale and shares the factor with the others
        float my_am = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float am = __uint_as_float(redux_max_u32(__float_as_uint(fabsf(v[j]))));
          my_am = (lane == j) ? am : my_am;
        }
        uint32_t my_code;
        float my_scale;
        block_scale<false>(my_am, norm, p.rcp_qmax, my_code, my_scale);
        uint8_t* const dcol = static_cast<uint8_t*>(p.d_col) + row * row_bytes + col_byte0;
        if (SCALAR) {
          // SCALAR (the 256-column backward epilogues): the 32 factors gathered
          // first; with them streamed those instances spill
#pragma unroll
          for (int j = 0; j < 32; ++j) sc[j] = __shfl_sync(0xffffffffu, my_scale, j);
          if (staged) store_q32_to<OUTC, false>(dcol_stage, v, sc, p.out_kind);
          else store_q32<OUTC, false>(dcol, v, sc, p.out_kind);
        } else {
          if (staged) store_q32_cols_to<OUTC>(dcol_stage, v, my_scale, p.out_kind);
          else store_q32_cols_to<OUTC>(dcol, v, my_scale, p.out_kind);
        }
        p.sfd_col[sf_off(col0 + lane, kblk_col, p.kq_col)] = static_cast<uint8_t>(my_code);
      } else {
        // FP4: each half-warp is one 16-row block (the whole warp one 32-row
        // block with one scale per 32 values).  Butterfly maxima inside the
        // half-warp; lane (16h + i) owns columns i and i + 16 of half h.
        const int h = lane >> 4, i = lane & 15;
        float am_lo = 0.0f, am_hi = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float m = fabsf(v[j]);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (j < 16) am_lo = (i == j) ? m : am_lo;
          else am_hi = (i == j - 16) ? m : am_hi;
        }
        if (v32) {
          am_lo = fmaxf(am_lo, __shfl_xor_sync(0xffffffffu, am_lo, 16));
          am_hi = fmaxf(am_hi, __shfl_xor_sync(0xffffffffu, am_hi, 16));
        }
        uint32_t code_lo, code_hi;
        float sc_lo, sc_hi;
        if (e4m3_sf) {
          block_scale<true>(am_lo, norm, p.rcp_qmax, code_lo, sc_lo);
          block_scale<true>(am_hi, norm, p.rcp_qmax, code_hi, sc_hi);
        } else {
          block_scale<false>(am_lo, norm, p.rcp_qmax, code_lo, sc_lo);
          block_scale<false>(am_hi, norm, p.rcp_qmax, code_hi, sc_hi);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          sc[j] = __shfl_sync(0xffffffffu, j < 16 ? sc_lo : sc_hi, 16 * h + (j & 15));
        if (staged) store_q32_to<OUTC, !SCALAR>(dcol_stage, v, sc, p.out_kind);
        else store_q32<OUTC, !SCALAR>(static_cast<uint8_t*>(p.d_col) + row * row_bytes + col_byte0, v, sc, p.out_kind);
        if (!v32 || h == 0) {
          const int kb = v32 ? kblk_col : 2 * kblk_col + h;   // row-block index
          p.sfd_col[sf_off(col0 + i, kb, p.kq_col)] = static_cast<uint8_t>(code_lo);
          p.sfd_col[sf_off(col0 + i + 16, kb, p.kq_col)] = static_cast<uint8_t>(code_hi);
        }
      }
    }
  }
  if (staged) {
    // the warp's 32 rows of the chunk (and of the D_col chunk) in one TMA store each
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(os.d, os.slot, store_x, row);
      if (OUTC != OUTC_FLOAT && p.want_col) tma_store_2d(os.d_col, os.slot + kStoreSlot / 2, store_x, row);
      bulk_commit();
    }
  }
}

// Adds the column sums of a warp's 32 x 32 chunk (lane = row, v[i] = column i)
// to dst[0..31]: five exchange-and-add rounds halve the columns each lane
// keeps (31 shuffles), after which lane l holds column l's sum; one coalesced
// atomic add per lane.  v is consumed.
__device__ __forceinline__ void add_column_sums32(float (&v)[32], float* dst, int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  atomicAdd(dst + lane, v[0]);
}

// Rowwise Hadamard output of one 32-column chunk of D of one row: each 16-value
// block of bf16-rounded D times H16 / 4 (H16 the Sylvester Hadamard matrix,
// entry (i, j) = (-1)^popcount(i & j): four in-register butterfly stages),
// stored as bf16 or quantized to NVFP4 with E4M3 scales per 16 under rnorm.
__device__ __forceinline__ void rht_chunk(const Params& p, const float (&v)[32], int row, int col0,
                                          float rnorm) {
  float y[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i & o) continue;
        const float a = y[16 * h + i], b = y[16 * h + i + o];
        y[16 * h + i] = a + b;
        y[16 * h + i + o] = a - b;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] *= 0.25f;
  if (p.rht_kind == OK_BF16) {
    store_h32(static_cast<uint16_t*>(p.rht) + static_cast<int64_t>(row) * p.n_out + col0, &y[0], OK_BF16);
  } else {
    float sc[32];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(y[16 * b + i]));
      uint32_t code;
      float s;
      block_scale<true>(am, rnorm, 1.0f / 6.0f, code, s);
#pragma unroll
      for (int i = 0; i < 16; ++i) sc[16 * b + i] = s;
      p.sfrht[sf_off(row, col0 / 16 + b, p.kq_rht)] = static_cast<uint8_t>(code);
    }
    store_q32<OUTC_FP4>(static_cast<uint8_t*>(p.rht) + static_cast<int64_t>(row) * (p.n_out / 2) + col0 / 2, y,
                        sc, OK_E2M1);
  }
}

// Colwise Hadamard output of one 32-column chunk of D held by a warp (lane =
// row): each half-warp's 16 rows are a block of 16 consecutive tokens of the
// expert whose padded rows start at seg_start (em of them).  Per column: bf16
// rounding, the 16-point transform across the half-warp's lanes (four xor
// butterfly stages, entry (i, j) of H16 = (-1)^popcount(i & j)) times 1/4, the
// block's E4M3 scale under rnorm, E2M1 codes paired by neighbouring lanes into
// bytes at flat element n_out * seg_start + column * em + token.
__device__ __forceinline__ void rht_col_chunk(const Params& p, const float (&v)[32], int row, int col0, int lane,
                                              int64_t seg_start, int em, float rnorm) {
  if constexpr (kDebugBounds) {
    if (__any_sync(0xffffffffu, !in_range(p.status, kSiteRht, seg_start + em - 1, p.m_pad))) return;
  }
  const int t = static_cast<int>(row - seg_start);     // token within the expert
  const int64_t seg_elem = static_cast<int64_t>(p.n_out) * seg_start;
  const int kq = (em / 16 + 3) / 4;                    // SF atoms per 128 columns of the segment
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float y = __bfloat162float(__float2bfloat16_rn(v[j]));
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const float other = __shfl_xor_sync(0xffffffffu, y, o);
      y = (lane & o) ? (other - y) : (y + other);
    }
    y *= 0.25f;
    float am = fabsf(y);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    uint32_t code;
    float s;
    block_scale<true>(am, rnorm, 1.0f / 6.0f, code, s);
    const float q = y * s;
    const float q_odd = __shfl_xor_sync(0xffffffffu, q, 1);
    const int n = col0 + j;
    if ((lane & 1) == 0) {
      const int64_t e = seg_elem + static_cast<int64_t>(n) * em + t;   // even: low nibble
      static_cast<uint8_t*>(p.rht)[e >> 1] = static_cast<uint8_t>(cvt_e2m1x2(q, q_odd));
    }
    if ((lane & 15) == 0) p.sfrht[seg_elem / 16 + sf_off(n, t / 16, kq)] = static_cast<uint8_t>(code);
  }
}

// Step 2 and Step 3 for one 32-column chunk of one row: C = al * xs (the
// input half for the GLUs; fp32 bits), al * gs the gate half.  al is alpha_g,
// or 1 where alpha and the bias were already applied in place.
template <int IC, int EPI, int OUTC, bool XC>
__device__ __forceinline__ void epilogue_chunk(const Params& p, const uint32_t* xs, const uint32_t* gs, int row,
                                               int col0, float al, float pr, float norm, int lane, int kblk_col,
                                               float& amax_local, int64_t seg_start, int seg_rows,
                                               const OutStage& os) {
  // two values per instruction where the arithmetic is a plain product or sum
  // (packed f32x2, the same IEEE round-to-nearest as the scalar operations)
  float v[32];
  const float2 al2 = make_float2(al, al), pr2 = make_float2(pr, pr);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 c = __fmul2_rn(al2, make_float2(__uint_as_float(xs[i]), __uint_as_float(xs[i + 1])));
    float2 o;
    if (EPI == EPI_GATE) {
      o = __fmul2_rn(pr2, c);
    } else if (EPI == EPI_SRELU) {
      float2 r = make_float2(fmaxf(c.x, 0.0f), fmaxf(c.y, 0.0f));
      if (p.tanh_s > 0.0f) {
        const float2 t = __fmul2_rn(r, make_float2(p.tanh_rcp_s, p.tanh_rcp_s));
        r = __fmul2_rn(make_float2(p.tanh_s, p.tanh_s),
                       make_float2(fminf(tanh_approx(t.x), 1.0f), fminf(tanh_approx(t.y), 1.0f)));
      }
      o = __fmul2_rn(pr2, __fmul2_rn(r, r));
    } else {
      // SwiGLU: X * G * sigmoid(G); GeGLU: (X + 1) * G * sigmoid(1.702 G); both
      // halves first clamped to [-glu_limit, glu_limit] when a limit is set
      float2 x = c;
      float2 gt = __fmul2_rn(al2, make_float2(__uint_as_float(gs[i]), __uint_as_float(gs[i + 1])));
      if (p.glu_limit > 0.0f) {
        x.x = fminf(fmaxf(x.x, -p.glu_limit), p.glu_limit);
        x.y = fminf(fmaxf(x.y, -p.glu_limit), p.glu_limit);
        gt.x = fminf(fmaxf(gt.x, -p.glu_limit), p.glu_limit);
        gt.y = fminf(fmaxf(gt.y, -p.glu_limit), p.glu_limit);
      }
      float2 sig;
      if (p.glu_kind) {
        sig.x = __fdividef(1.0f, 1.0f + __expf(-1.702f * gt.x));
        sig.y = __fdividef(1.0f, 1.0f + __expf(-1.702f * gt.y));
        o = __fmul2_rn(__fmul2_rn(pr2, __fadd2_rn(x, make_float2(1.0f, 1.0f))), __fmul2_rn(gt, sig));
      } else {
        sig.x = __fdividef(1.0f, 1.0f + __expf(-gt.x));
        sig.y = __fdividef(1.0f, 1.0f + __expf(-gt.y));
        o = __fmul2_rn(__fmul2_rn(pr2, x), __fmul2_rn(gt, sig));
      }
      if (p.glu_gamma != 1.0f) o = __fmul2_rn(o, make_float2(p.glu_gamma, p.glu_gamma));
    }
    v[i] = o.x;
    v[i + 1] = o.y;
  }
  output_chunk<IC, OUTC>(p, v, row, col0, norm, lane, kblk_col, amax_local, os);
  if (XC && p.rht != nullptr && in_range(p.status, kSiteRht, col0 + 31, p.n_out)) {
    if (p.rht_colwise) rht_col_chunk(p, v, row, col0, lane, seg_start, seg_rows, *p.rht_norm_const);
    else rht_chunk(p, v, row, col0, *p.rht_norm_const);
  }
}

// XC: a forward launch adds a bias to C, stores C or writes the Hadamard
// output; a backward launch accumulates dbias (separate instances, so that the
// register budget of the plain epilogue is untouched).
template <int IC, int BN, int CM, int EPI, int OUTC, bool XC>
__global__ void __launch_bounds__(Roles<scale_stores<ic_fp4(IC)>()>::kThreads, 1)
    bsgg_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmDcol,
                const __grid_constant__ Params p) {
  constexpr bool FP4 = ic_fp4(IC);
  constexpr bool SCALED = ic_scaled(IC);
  constexpr bool PAIR = CM == CM_PAIR;
  constexpr bool CLUSTER = CM != CM_SINGLE;
  constexpr bool ST = scale_stores<FP4>();
  using Ro = Roles<ST>;
  using Ly = Layout<FP4, BN, PAIR, SCALED, stage_slices(IC, CM)>;
  constexpr int S = Ly::kStages;
  constexpr int NA = Ly::kNumAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Ly::kOffBars;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S + NA + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * NA);
  // stage's scale atoms are in tensor memory (and so its operands in shared memory)
  auto sfr_bar = [&](int st) { return bar0 + 8u * (2 * S + 2 * NA + 1 + st); };
  const uint32_t drain_bar2 = bar0 + 8u * (3 * S + 2 * NA + 1);   // the scale copier's own drain
  // pairs storing scales: this CTA's scale atoms of the stage have landed (the
  // operands complete the even CTA's "full" barrier, the scales their own CTA's)
  auto sfull_bar = [&](int st) { return bar0 + 8u * (3 * S + 2 * NA + 2 + st); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Ly::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kOffAbort);
  int32_t* s_trow = reinterpret_cast<int32_t*>(smem + Ly::kOffTrows);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + Ly::kOffOffsets);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  const bool issues_mma = !PAIR || leader;       // the CTA that issues this CTA's MMAs and copies
  const int unit = CLUSTER ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int num_units = CLUSTER ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  for (int i = tid; i < p.L; i += Ro::kThreads) s_off[i] = p.offsets[i];
  if (tid == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int a = 0; a < NA; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    // stores: the four scale warps of each CTA report to the even CTA
    for (int st = 0; st < S; ++st) mbar_init(sfr_bar(st), ST ? (PAIR ? 8 : 4) : 1);
    for (int st = 0; st < S; ++st) mbar_init(sfull_bar(st), 1);
    mbar_init(drain_bar2, 1);
    *abort_flag = 0;
    mbar_fence_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (SCALED) {
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) {
    if (PAIR) { tmem_alloc_pair(smem_u32(tmem_holder), Ly::kTmemCols); tmem_relinquish_pair(); }
    else { tmem_alloc(smem_u32(tmem_holder), Ly::kTmemCols); tmem_relinquish(); }
  }
  tc_fence_before();
  if (CLUSTER) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // padded_offsets must be non-decreasing multiples of 128 ending at m_pad.
  int bad = 0;
  for (int i = tid; i < p.L; i += Ro::kThreads) {
    const int prev = i ? s_off[i - 1] : 0;
    if (s_off[i] < prev || (s_off[i] % kBM) != 0) bad = 1;
  }
  if (tid == 0 && s_off[p.L - 1] != p.m_pad) bad = 1;
  if (tid == 0 && p.b_maps != nullptr && *p.maps_bad != 0u) bad = 1;   // discrete mode: bad pointers
  bad = __syncthreads_or(bad);
  // tile rows per group, inclusive prefix (warp 0: contiguous chunks per lane)
  if (!bad && warp == 0) {
    const int chunk = (p.L + 31) / 32;
    const int g0 = lane * chunk, g1 = min(p.L, g0 + chunk);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int mt = (s_off[g] - (g ? s_off[g - 1] : 0)) / kBM;
      local += group_units<CM>(mt);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int g = g0; g < g1; ++g) {
      const int mt = (s_off[g] - (g ? s_off[g - 1] : 0)) / kBM;
      run += group_units<CM>(mt);
      s_trow[g] = run;
    }
  }
  __syncthreads();
  const int num_tiles = bad ? 0 : s_trow[p.L - 1] * p.num_n_tiles;

  if (bad) {
    // (bad pointers were reported by the kernel that wrote the maps)
    if (blockIdx.x == 0 && tid == 0 && !(p.b_maps != nullptr && *p.maps_bad != 0u))
      atomicOr(p.status, kStatusBadOffsets);
  } else if (ST ? warp < 8 : (warp < 2 || warp == Ro::kCopyWarp)) {
    // producer, MMA issuer, scale warps (and, storing scales, two idle warps)
    if constexpr (ST) setmaxnreg_dec<Ro::kLowRegs>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_phase[S];
        bool issued[S];
#pragma unroll
        for (int s = 0; s < S; ++s) { issued[s] = false; issued_phase[s] = 0; }
        bool ok = true;
        int fenced_g = -1;
        for (int t = unit; t < num_tiles && ok; t += num_units) {
          int g, mt, nt;
          bool valid;
          decode_tile<CM>(t, p, s_off, s_trow, rank, g, mt, nt, valid);
          const int b_row = nt * BN + (PAIR ? static_cast<int>(rank) * Ly::kBRows : 0);
          // dense weights: expert g is slice g of B and of SFB; discrete weights:
          // expert g's own maps, each of one slice
          const CUtensorMap* mB = &tmB;
          const CUtensorMap* mSFB = &tmSFB;
          int bz = g, sfb_rb = g * p.rn_b + nt * Ly::kHalves;
          if (p.b_maps != nullptr) {
            mB = p.b_maps + 2 * g;
            mSFB = mB + 1;
            bz = 0;
            sfb_rb = nt * Ly::kHalves;
            if (g != fenced_g) {
              tmap_acquire(mB);
              if (SCALED) tmap_acquire(mSFB);
              fenced_g = g;
            }
          }
          for (int ks = 0; ks < p.num_k_stages; ++ks) {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns)) { ok = false; break; }
            const uint32_t fb = full_bar(stage);
            // scale atoms this stage loads (FP4 with one scale per 32 values: half)
            const int atoms_ld = IC == IC_F4E8 ? p.sf_atoms : Ly::kAtoms;
            const uint32_t sf_tx = static_cast<uint32_t>(atoms_ld * 512 * (1 + Ly::kHalves));
            const int k0 = ks * Ly::kStageK, ka = 2 * ks * atoms_ld;
            // the K slices of this stage inside K (a two-slice stage at the K
            // tail may hold only its first); a slice is one box per operand
            const int kb_bytes = !SCALED ? 2 * p.k : FP4 ? p.k / 2 : p.k;
            const int nsl = (Ly::kSlices == 1 || k0 + kBKBytes < kb_bytes) ? Ly::kSlices : 1;
            const uint32_t op_tx = static_cast<uint32_t>(nsl * (Ly::kASlice + Ly::kBSlice));
            const uint32_t sA = sbase + Ly::kOffA + stage * Ly::kABytes;
            const uint32_t sB = sbase + Ly::kOffB + stage * Ly::kBBytes;
            const uint32_t sSa = sbase + Ly::kOffSfa + stage * Ly::kSfaBytes;
            const uint32_t sSb = sbase + Ly::kOffSfb + stage * Ly::kSfbBytes;
            if constexpr (kDebugBounds) {
              // box origins: A's 128 rows, the K byte offset, B's n-tile and
              // slice (a B box may start or run past N: those rows are
              // zero-filled and their columns are not stored), the
              // scale boxes' atom row and first 128-row block, inside the
              // expert's blocks (with N not a multiple of the tile the SFB box
              // runs on into the next expert's blocks or past the end: those
              // rows' B data is zero-filled and their columns are not stored)
              const int v = !FP4 ? 32 : (IC == IC_F4E8 && p.sf_v32) ? 32 : 16;
              const int kq = ((p.k + v - 1) / v + 3) / 4;
              const int slices = p.b_maps != nullptr ? 1 : p.L;
              bool in = in_range(p.status, kSiteARows, mt * kBM + kBM - 1, p.dbg_rows) &&
                        in_range(p.status, kSiteK, k0, kb_bytes) && in_range(p.status, kSiteBRow, nt, p.num_n_tiles) &&
                        in_range(p.status, kSiteBSlice, bz, slices);
              if (SCALED)
                in = in && in_range(p.status, kSiteSfa, ka, 2 * kq) &&
                     in_range(p.status, kSiteSfb, nt * Ly::kHalves, p.rn_b) &&
                     in_range(p.status, kSiteSfb, sfb_rb, p.rn_b * slices);
              if (!in) {
                *abort_flag = 1;
                ok = false;
                break;
              }
            }
            if (PAIR && ST) {
              // both CTAs' operand bytes complete the even CTA's barrier, each
              // CTA's scale bytes its own (its scale warps wait there)
              const uint32_t fbl = mapa_shared(fb, 0);
              const uint32_t sfb_own = sfull_bar(stage);
              if (leader) mbar_expect_tx(fb, 2u * op_tx);
              mbar_expect_tx(sfb_own, sf_tx);
              // the scales first: the scale warps' stores into tensor memory
              // follow their arrival, the MMAs wait for both
              tma_load_3d(sSb, mSFB, sfb_own, 0, ka, sfb_rb);
              tma_load_3d(sSa, &tmSFA, sfb_own, 0, ka, mt);
              for (int j = 0; j < nsl; ++j) {
                tma_load_2d_pair(sA + j * Ly::kASlice, &tmA, fbl, k0 + j * kBKBytes, mt * kBM);
                tma_load_3d_pair(sB + j * Ly::kBSlice, mB, fbl, k0 + j * kBKBytes, b_row, bz);
              }
            } else if (PAIR) {
              // both CTAs' bytes complete the even CTA's barrier
              const uint32_t fbl = mapa_shared(fb, 0);
              if (leader) mbar_expect_tx(fb, 2u * (op_tx + (SCALED ? sf_tx : 0u)));
              for (int j = 0; j < nsl; ++j) {
                tma_load_2d_pair(sA + j * Ly::kASlice, &tmA, fbl, k0 + j * kBKBytes, mt * kBM);
                tma_load_3d_pair(sB + j * Ly::kBSlice, mB, fbl, k0 + j * kBKBytes, b_row, bz);
              }
              if (SCALED) {
                tma_load_3d_pair(sSa, &tmSFA, fbl, 0, ka, mt);
                tma_load_3d_pair(sSb, mSFB, fbl, 0, ka, sfb_rb);
              }
            } else {
              mbar_expect_tx(fb, op_tx + (SCALED ? sf_tx : 0u));
              for (int j = 0; j < nsl; ++j) {
                tma_load_2d(sA + j * Ly::kASlice, &tmA, fb, k0 + j * kBKBytes, mt * kBM);
                tma_load_3d(sB + j * Ly::kBSlice, mB, fb, k0 + j * kBKBytes, b_row, bz);
              }
              if (SCALED) {
                tma_load_3d(sSa, &tmSFA, fb, 0, ka, mt);
                tma_load_3d(sSb, mSFB, fb, 0, ka, sfb_rb);
              }
            }
            issued[stage] = true;
            issued_phase[stage] = phase;
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
        if (ok && CLUSTER) {
          // wait until the last use of every stage was released: no commit or
          // MMA read of the even CTA still targets this CTA's shared memory when
          // the CTAs part
          for (int i = 0; i < S; ++i) {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns)) { ok = false; break; }
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          // drain: wait (bounded) for every load this thread issued to land.  In a
          // pair the loads also complete the even CTA's barriers, which cannot be
          // polled from here: wait out the drain bound instead.
          for (int s = 0; s < S; ++s)
            if (issued[s]) {
              const uint64_t t0 = globaltimer_ns();
              while (globaltimer_ns() - t0 < kDrainLimitNs) {
                if (!CLUSTER && mbar_try_wait(full_bar(s), issued_phase[s])) break;
              }
              if (CLUSTER) break;
            }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // One thread issues every tcgen05 operation of the CTA (pair).  Its loop is
      // kept short: the tcgen05 queue holds little more than one stage, so any
      // per-MMA scalar work would leave the tensor pipe idle.  All shared-memory
      // descriptors are formed once and advanced by adds (the start-address field
      // holds address / 16 in its low 14 bits; every address here is < 256 KB).
      if (lane == 0 && issues_mma) {
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        const uint32_t sf_tmem0 = tmem_base + NA * BN;
        const uint64_t a_desc0 = sdesc_kmajor_sw128(sbase + Ly::kOffA);
        const uint64_t b_desc0 = sdesc_kmajor_sw128(sbase + Ly::kOffB);
        // instruction descriptors of the four MMAs of a stage: MXFP8 selects the
        // scale byte (k-block) of each row's word, NVFP4 uses whole words
        uint32_t idk[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          idk[kk] = (FP4 || !SCALED) ? p.idesc
                                     : (p.idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4));
        const int full_stages = p.k / Ly::kKElems;      // stages with all of their MMAs
        auto issue_stage = [&](uint32_t d_tmem, int st, int n_mma, uint32_t acc0) {
          const uint32_t sfa_t = sf_tmem0 + st * Ly::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + Ly::kSfaCols;
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((st * Ly::kABytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((st * Ly::kBBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < Ly::kMmas; ++kk) {
            if (kk >= n_mma) break;
            const uint32_t accum = kk ? 1u : acc0;
            // MMA kk reads K bytes [32 (kk % 4), + 32) of slice kk / 4: +2 in
            // descriptor units per MMA, a slice's bytes / 16 per slice
            const int sl = kk / 4, kq = kk % 4;
            const uint64_t adk = ad + static_cast<uint64_t>(sl * (Ly::kASlice >> 4) + 2 * kq);
            const uint64_t bdk = bd + static_cast<uint64_t>(sl * (Ly::kBSlice >> 4) + 2 * kq);
            if (!SCALED) {
              if (PAIR) tc_mma_bf16_pair(d_tmem, adk, bdk, idk[kq], accum);
              else tc_mma_bf16(d_tmem, adk, bdk, idk[kq], accum);
            } else if (FP4) {
              // one scale atom per MMA
              const uint32_t sa = sfa_t + 4 * kk, sb = sfb_t + 4 * Ly::kHalves * kk;
              if (PAIR) tc_mma_nvf4_pair(d_tmem, adk, bdk, idk[kq], sa, sb, accum);
              else tc_mma_nvf4(d_tmem, adk, bdk, idk[kq], sa, sb, accum);
            } else {
              // one scale atom per slice, the instruction descriptor selects its byte
              const uint32_t sa = sfa_t + 4 * sl, sb = sfb_t + 4 * Ly::kHalves * sl;
              if (PAIR) tc_mma_mxf8_pair(d_tmem, adk, bdk, idk[kq], sa, sb, accum);
              else tc_mma_mxf8(d_tmem, adk, bdk, idk[kq], sa, sb, accum);
            }
          }
          // release the stage (in both CTAs of a cluster)
          if (PAIR) tc_commit_pair(empty_bar(st), 3);
          else tc_commit(empty_bar(st));
        };
        // failure-path test: nothing arrives on the drain barrier before an abort
        if (p.force_timeout && !mbar_wait(drain_bar, 0, abort_flag, p.wait_limit_ns)) ok = false;
        for (int t = unit; t < num_tiles && ok; t += num_units) {
          if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.wait_limit_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int ks = 0; ks < p.num_k_stages; ++ks) {
            // pairs storing scales: the scale warps waited for the scales only
            if (PAIR && ST && !mbar_wait(full_bar(stage), phase, abort_flag, p.wait_limit_ns)) { ok = false; break; }
            // the stage's operands (and scales, through the scale warp or copier)
            const uint32_t ready = SCALED ? sfr_bar(stage) : full_bar(stage);
            if (!mbar_wait(ready, phase, abort_flag, p.wait_limit_ns)) { ok = false; break; }
            tc_fence_after();
            if (ks < full_stages) {
              issue_stage(d_tmem, stage, Ly::kMmas, ks ? 1u : 0u);
            } else {
              const int k_left = p.k - ks * Ly::kKElems;
              issue_stage(d_tmem, stage, (k_left + Ly::kMmaK - 1) / Ly::kMmaK, ks ? 1u : 0u);
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          if (PAIR) tc_commit_pair(accf_bar(acc), 3); else tc_commit(accf_bar(acc));
          if (++acc == NA) { acc = 0; acc_phase ^= 1u; }
        }
        if (!ok) {
          atomicOr(p.status, kStatusTimeout);
          // drain: wait (bounded) until every issued tcgen05 operation completed
          if (PAIR) tc_commit_pair(drain_bar, 1); else tc_commit(drain_bar);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < kDrainLimitNs) {}
        }
      }
    } else if (ST ? warp < 6 : true) {
      if constexpr (ST) {
        // ------------------------------------------------------------ scale stores
        // One warp per tensor-memory lane quadrant q.  The MMA reads row r's A
        // scales from lane r, column (r / 32) % 4 of the atom's 4-column group, so
        // the warp writes A's atoms into column q of its own 32 lanes only; every
        // quadrant reads the scales of every B row, so B's atoms go into all four
        // columns.  A quarter of A's tensor-memory writes of the copy path.
        const uint32_t q = static_cast<uint32_t>(warp & 3);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint32_t sf_tmem0 = tmem_base + NA * BN + ((q * 32u) << 16);
        for (int t = unit; t < num_tiles && ok; t += num_units) {
          for (int ks = 0; ks < p.num_k_stages; ++ks) {
            const uint32_t landed = PAIR ? sfull_bar(stage) : full_bar(stage);
            if (!__all_sync(0xffffffffu, mbar_wait(landed, phase, abort_flag, p.wait_limit_ns))) {
              ok = false;
              break;
            }
            const uint32_t slot = sf_tmem0 + stage * Ly::kSfColsPerStage;
            const uint8_t* sa = smem + Ly::kOffSfa + stage * Ly::kSfaBytes + 16 * lane;
            const uint8_t* sb = smem + Ly::kOffSfb + stage * Ly::kSfbBytes + 16 * lane;
            if (IC != IC_F4E8 || p.sf_atoms == Ly::kAtoms) {
              // sixteen columns per store: A's atoms whole (the 16 bytes a
              // lane holds are rows lane + 32j; quadrant q's MMA rows read
              // column q of each atom's group, the other three are not read
              // by them), then B's atoms in the column order 4 (i * halves + h)
              static_assert(Ly::kAtoms == 4, "four scale atoms per stage and 128 rows");
              uint4 v[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4*>(sa + 512 * i);
              tmem_st_x16(slot, v);
#pragma unroll
              for (int c0 = 0; c0 < 4 * Ly::kHalves; c0 += 4) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int i = (c0 + k) / Ly::kHalves, h = (c0 + k) % Ly::kHalves;
                  v[k] = *reinterpret_cast<const uint4*>(sb + 512 * (h * Ly::kAtoms + i));
                }
                tmem_st_x16(slot + Ly::kSfaCols + 4 * c0, v);
              }
            } else {
              // one scale per 32 values: a loaded word [s0 s1 s2 s3] covers two
              // MMAs; the MMA's 16-value slots get [s0 s0 s1 s1] and [s2 s2 s3 s3]
              // (the same products as one scale per 32 values)
              constexpr int kSrc = Ly::kAtoms / 2;
#pragma unroll
              for (int i = 0; i < Ly::kAtoms; ++i) {
                const uint32_t sel = (i & 1) ? 0x3322u : 0x1100u;
                const uint4 va = *reinterpret_cast<const uint4*>(sa + 512 * (i / 2));
                const uint32_t wa = q == 0 ? va.x : q == 1 ? va.y : q == 2 ? va.z : va.w;
                tmem_st_x1(slot + 4 * i + q, __byte_perm(wa, 0u, sel));
#pragma unroll
                for (int h = 0; h < Ly::kHalves; ++h) {
                  const uint4 vb = *reinterpret_cast<const uint4*>(sb + 512 * (h * kSrc + i / 2));
                  tmem_st_x4(slot + Ly::kSfaCols + 4 * (i * Ly::kHalves + h),
                             make_uint4(__byte_perm(vb.x, 0u, sel), __byte_perm(vb.y, 0u, sel),
                                        __byte_perm(vb.z, 0u, sel), __byte_perm(vb.w, 0u, sel)));
                }
              }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR) mbar_arrive_cluster(mapa_shared(sfr_bar(stage), 0));
              else mbar_arrive(sfr_bar(stage));
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok && lane == 0) atomicOr(p.status, kStatusTimeout);
      } else {
        // ------------------------------------------------------------ scale copier
        // Same stage sequence as the MMA issuer.  Writing a stage's tensor-memory
        // scale slot is safe once its "full" barrier completed: the refill behind
        // it waited for the MMAs that read the slot's previous contents.
        // (bfloat16 operands have no scales: the MMA issuer waits on "full".)
        if (SCALED && lane == 0 && issues_mma) {
          int stage = 0;
          uint32_t phase = 0;
          bool ok = true;
          const uint32_t sf_tmem0 = tmem_base + NA * BN;
          const uint64_t sfa_desc0 = sdesc_sf_block(sbase + Ly::kOffSfa);
          const uint64_t sfb_desc0 = sdesc_sf_block(sbase + Ly::kOffSfb);
          for (int t = unit; t < num_tiles && ok; t += num_units) {
            for (int ks = 0; ks < p.num_k_stages; ++ks) {
              if (!mbar_wait(full_bar(stage), phase, abort_flag, p.wait_limit_ns)) { ok = false; break; }
              tc_fence_after();
              const uint32_t sfa_t = sf_tmem0 + stage * Ly::kSfColsPerStage;
              const uint32_t sfb_t = sfa_t + Ly::kSfaCols;
              const uint64_t sfa_d = sfa_desc0 + static_cast<uint64_t>((stage * Ly::kSfaBytes) >> 4);
              const uint64_t sfb_d = sfb_desc0 + static_cast<uint64_t>((stage * Ly::kSfbBytes) >> 4);
              // atom i of A at columns 4i; atom i of B's 128-row block h at
              // columns 4 * (i * halves + h)
#pragma unroll
              for (int i = 0; i < Ly::kAtoms; ++i) {
                if (PAIR) tc_cp_32x128b_x4_pair(sfa_t + 4 * i, sfa_d + 32 * i);
                else tc_cp_32x128b_x4(sfa_t + 4 * i, sfa_d + 32 * i);
#pragma unroll
                for (int h = 0; h < Ly::kHalves; ++h) {
                  const uint32_t dst = sfb_t + 4 * (i * Ly::kHalves + h);
                  const uint64_t src = sfb_d + 32 * (h * Ly::kAtoms + i);
                  if (PAIR) tc_cp_32x128b_x4_pair(dst, src); else tc_cp_32x128b_x4(dst, src);
                }
              }
              if (PAIR) tc_commit_pair(sfr_bar(stage), 1); else tc_commit(sfr_bar(stage));
              if (++stage == S) { stage = 0; phase ^= 1u; }
            }
          }
          if (!ok) {
            atomicOr(p.status, kStatusTimeout);
            // drain: wait (bounded) until this thread's copies completed
            if (PAIR) tc_commit_pair(drain_bar2, 1); else tc_commit(drain_bar2);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain_bar2, 0) && globaltimer_ns() - t0 < kDrainLimitNs) {}
          }
        }
      }
    }
  } else {
    if constexpr (ST) setmaxnreg_inc<Ro::kHighRegs>();
    // ------------------------------------------------------------ epilogue
    constexpr int kWarpCols = BN / 2;                 // accumulator columns per warp
    // 256-column tiles with two accumulators (bfloat16 operands, no scale
    // slots): the warp reads its columns 32 at a time as it uses them and hands
    // the accumulator back at the end of the tile, while the MMAs fill the
    // other one.  Holding all 128 in registers spills the backward epilogue.
    constexpr bool kChunkLd = NA == 2 && BN == 256;
    static_assert(!kChunkLd || is_bwd_inst(EPI), "chunked accumulator reads: backward epilogues");
    // the forward GLU pairs its up and gate blocks as it reads the accumulator
    // (the bias / C instances keep the accumulator's column order in registers)
    constexpr bool kPairOnLoad = EPI == EPI_SWIGLU && !XC;
    // the backward's arithmetic and quantization packed two values per
    // instruction on 128-column tiles and where the accumulator is read 32
    // columns at a time (the other 256-column backward instances spill with
    // the packed form and keep the scalar one)
    constexpr bool kPackedBwd = is_bwd_inst(EPI) && (BN == 128 || kChunkLd);
    const int q = warp & 3;                           // tensor-memory lane quadrant
    const int e = (warp - Ro::kEpiFirst) >> 2;        // which half of the columns
    const float norm = (OUTC == OUTC_FLOAT) ? 1.0f : *p.norm_const;
    // D (and D_col) through this warp's staging slot and TMA stores where the
    // layout has room for the slots and the chunk is not fp32 (MXFP8 and
    // bfloat16 inputs; measured FC1 +0.8 %, FC2 +1.8 %, skewed +0.9 %)
    const OutStage os{(!FP4 && Ly::kTmaStore && !(OUTC == OUTC_FLOAT && p.out_kind == OK_F32))
                          ? sbase + Ly::kOffStore + static_cast<uint32_t>((warp - Ro::kEpiFirst) * kStoreSlot)
                          : 0u,
                      &tmD, &tmDcol};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit; t < num_tiles; t += num_units) {
      int g, mt, nt;
      bool valid;
      decode_tile<CM>(t, p, s_off, s_trow, rank, g, mt, nt, valid);
      // dSwiGLU backward: the saved-C values this thread will read are fetched
      // into L2 while the tile's MMAs run (+3.6 % on the FC1 backward).  Holding
      // them in registers instead spills the epilogue to local memory, which
      // misses L1 here (nearly all of it is shared memory): 43 % slower.
      if (is_bwd_inst(EPI) && valid) {
        // the saved-C values this thread will read, fetched into L2 while the
        // tile's MMAs run: 2 * kWarpCols values of its row from column
        // 2 * (first GEMM column of its half)
        const int j0 = nt * BN + e * kWarpCols;
        if (j0 < p.n) {
          const int esz = p.saved_c_kind == OK_F32 ? 4 : 2;
          const uint8_t* base = static_cast<const uint8_t*>(p.saved_c) +
                                ((static_cast<int64_t>(mt * kBM + q * 32 + lane) * 2 * p.n + 2 * j0) * esz);
          const int bytes = 2 * min(kWarpCols, p.n - j0) * esz;
          for (int o = 0; o < bytes; o += 128) prefetch_l2(base + o);
        }
      }
      const bool got = __all_sync(0xffffffffu, mbar_wait(accf_bar(acc), acc_phase, abort_flag, p.wait_limit_ns));
      if (!got) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      uint32_t r[kWarpCols];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + e * kWarpCols;
      const int acc_cur = acc;
      auto release = [&]() {
        // this warp is done with the accumulator: hand it back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) mbar_arrive_cluster(mapa_shared(acce_bar(acc_cur), 0));
          else mbar_arrive(acce_bar(acc_cur));
        }
      };
      if (!kChunkLd) {
        // SwiGLU / GeGLU without bias or C: each 64-column pair's up block is
        // read into its first 32 registers and its gate block into the next 32,
        // whichever comes first in the accumulator (gate_first)
        const uint32_t swap = (kPairOnLoad && p.gate_first) ? 32u : 0u;
#pragma unroll
        for (int c = 0; c < kWarpCols / 32; ++c) tmem_ld32p(taddr + ((32u * c) ^ swap), &r[32 * c]);
        tmem_wait_ld();
        release();       // all of this warp's columns are in registers
      }
      if (++acc == NA) { acc = 0; acc_phase ^= 1u; }
      if (!valid) {
        if (kChunkLd) release();
        continue;
      }
      if constexpr (kDebugBounds) {
        // the rows of prob / D / dprob this warp touches and the group of alpha, bias, amax
        const bool in = in_range(p.status, kSiteDRow, mt * kBM + q * 32 + lane, p.dbg_rows) &&
                        in_range(p.status, kSiteGroup, g, p.L);
        if (__any_sync(0xffffffffu, !in)) {
          if (kChunkLd) release();
          continue;
        }
      }
      const int row = mt * kBM + q * 32 + lane;
      const float pr = p.prob[row];
      const float al = p.alpha[g];
      const int kblk_col = mt * 4 + q;                // this warp's 32-row block
      const int64_t seg_start = g ? s_off[g - 1] : 0;  // the group's padded rows (colwise RHT)
      const int seg_rows = static_cast<int>(s_off[g] - seg_start);
      // With a bias or a C output: C = alpha_g * acc + bias_g[n] in place (then
      // al = 1), stored when asked for ("Grouped GEMM + GLU + Hadamard + Quant
      // (SM100)", Equations)
      float al_epi = al;
      if (XC && (p.bias != nullptr || p.c_out != nullptr)) {
        const int ccol0 = nt * BN + e * kWarpCols;    // first C column of this warp's half
#pragma unroll
        for (int c = 0; c < kWarpCols / 32; ++c) {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[32 * c + i] = __float_as_uint(al * __uint_as_float(r[32 * c + i]));
          const int col0 = ccol0 + 32 * c;
          if (col0 < p.n) {
            if (p.bias != nullptr) {
              const int esz = p.bias_kind == OK_F32 ? 4 : 2;
              add_bias32(&r[32 * c],
                         static_cast<const uint8_t*>(p.bias) + (static_cast<int64_t>(g) * p.n + col0) * esz,
                         p.bias_kind);
            }
            if (p.c_out != nullptr && in_range(p.status, kSiteC, col0 + 31, p.n)) store_c32(p, &r[32 * c], row, col0);
          }
        }
        al_epi = 1.0f;
      }
      float amax_local = 0.0f;
      float amax_local2 = 0.0f;                       // backward: the gate-gradient blocks
      if (is_bwd_inst(EPI)) {
        // dSwiGLU backward ("Grouped GEMM + dGLU (SM100)", Block-scaled contract):
        // GEMM column j of pair b = j / 32 -> D (and saved C) columns 64b + r of
        // the input block and of the gate block, in the forward's block order
        // beta scales the saved C for dSwiGLU, and for dGeGLU on bfloat16
        // operands (the BF16 contract's X = beta C)
        const float al2 = al * al,
                    bt = (EPI == EPI_DSWIGLU && (p.bwd_kind == 0 || IC == IC_BF16)) ? p.beta[g] : 1.0f;
        const bool gf = p.gate_first != 0;
        float dprob_local = 0.0f;
        // chunked reads: one 32-column buffer; with dbias the loop stays rolled
        // (unrolled, that instance spills 7 KB)
        uint32_t rbuf[32];
#pragma unroll((kChunkLd && XC) ? 1 : kWarpCols / 32)
        for (int c = 0; c < kWarpCols / 32; ++c) {
          const int j0 = nt * BN + e * kWarpCols + 32 * c;
          if (j0 >= p.n) continue;
          if (kChunkLd) {
            tmem_ld32p(taddr + 32 * c, rbuf);
            tmem_wait_ld();
          }
          const uint32_t* rc = kChunkLd ? rbuf : &r[32 * c];
          const int xo = 2 * j0 + (gf ? 32 : 0), go = 2 * j0 + (gf ? 0 : 32);
          float x[32], gv[32];
          const int64_t srow = static_cast<int64_t>(row) * 2 * p.n;
          const int esz = p.saved_c_kind == OK_F32 ? 4 : 2;
          load_f32x32(x, static_cast<const uint8_t*>(p.saved_c) + (srow + xo) * esz, p.saved_c_kind);
          load_f32x32(gv, static_cast<const uint8_t*>(p.saved_c) + (srow + go) * esz, p.saved_c_kind);
          if (EPI == EPI_DSWIGLU && p.bwd_kind == 0 && kPackedBwd) {
            // the same arithmetic two values per instruction (packed f32x2)
            const float2 al2v = make_float2(al2, al2), btv = make_float2(bt, bt), prv = make_float2(pr, pr);
            const float2 one = make_float2(1.0f, 1.0f);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 ref = __fmul2_rn(al2v, make_float2(__uint_as_float(rc[i]), __uint_as_float(rc[i + 1])));
              const float2 X = __fmul2_rn(btv, make_float2(x[i], x[i + 1]));
              const float2 G = __fmul2_rn(btv, make_float2(gv[i], gv[i + 1]));
              const float2 sg = make_float2(__fdividef(1.0f, 1.0f + __expf(-G.x)), __fdividef(1.0f, 1.0f + __expf(-G.y)));
              const float2 sw = __fmul2_rn(G, sg);
              const float2 dp = __fmul2_rn(__fmul2_rn(X, sw), ref);
              dprob_local += dp.x;                                      // dprob += X swish(G) ref
              dprob_local += dp.y;
              const float2 rp = __fmul2_rn(ref, prv);
              const float2 dx = __fmul2_rn(rp, sw);                     // d input
              const float2 dg = __fmul2_rn(__fmul2_rn(__fmul2_rn(rp, X), sg),
                                           __ffma2_rn(G, __fadd2_rn(one, make_float2(-sg.x, -sg.y)), one));   // d gate
              x[i] = dx.x;
              x[i + 1] = dx.y;
              gv[i] = dg.x;
              gv[i + 1] = dg.y;
            }
          } else if (EPI == EPI_DSWIGLU && p.bwd_kind == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float ref = al2 * __uint_as_float(rc[i]);
              const float X = bt * x[i], G = bt * gv[i];
              const float sg = __fdividef(1.0f, 1.0f + __expf(-G));
              const float sw = G * sg;
              dprob_local += X * sw * ref;                              // dprob += X swish(G) ref
              x[i] = ref * pr * sw;                                     // d input
              gv[i] = ref * pr * X * sg * (1.0f + G * (1.0f - sg));     // d gate
            }
          } else if (EPI == EPI_DSITUGLU) {
            // dSiTU-GLU: T_g = b1 tanh(G/b1) sigmoid(G), T_u = b2 tanh(U/b2).
            // tanhf, not the approximate instruction (its 2^-11 error would flip
            // quantized codes far more often than rounding does), and
            // 1 - tanh^2(y) as sech^2(y) = 4e / (1 + e)^2 with e = exp(-2|y|),
            // which keeps its relative precision where tanh^2 rounds to 1
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float ref = al2 * __uint_as_float(rc[i]);
              const float U = x[i], G = gv[i];
              const float yg = G / p.situ_b1, yu = U / p.situ_b2;
              const float thg = tanhf(yg), thu = tanhf(yu);
              const float eg = __expf(-2.0f * fabsf(yg)), eu = __expf(-2.0f * fabsf(yu));
              const float sech2_g = __fdividef(4.0f * eg, (1.0f + eg) * (1.0f + eg));
              const float sech2_u = __fdividef(4.0f * eu, (1.0f + eu) * (1.0f + eu));
              const float sg = __fdividef(1.0f, 1.0f + __expf(-G));
              const float tg = p.situ_b1 * thg * sg, tu = p.situ_b2 * thu;
              const float dtg = sech2_g * sg + p.situ_b1 * thg * sg * (1.0f - sg);
              const float dtu = sech2_u;
              dprob_local += ref * tg * tu;                             // dprob += ref T_g T_u
              x[i] = ref * pr * tg * dtu;                               // d up
              gv[i] = ref * pr * tu * dtg;                              // d gate
            }
          } else {
            // dGeGLU: the gate clamped above, the up value both ways; each
            // gradient masked where its own raw value lies beyond a bound.
            // bfloat16 operands: of beta C (the BF16 contract's X = beta C)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float ref = al2 * __uint_as_float(rc[i]);
              const float U = IC == IC_BF16 ? bt * x[i] : x[i], G = IC == IC_BF16 ? bt * gv[i] : gv[i];
              const float gc = fminf(G, p.clamp_max);
              const float uc = fminf(fmaxf(U, p.clamp_min), p.clamp_max);
              const float sg = __fdividef(1.0f, 1.0f + __expf(-p.geglu_a * gc));
              const float t = gc * sg;
              const float uo = uc + p.lin_offset;
              dprob_local += ref * t * uo;                              // dprob += ref Gc s (Uc + offset)
              // the masks multiply, as the page writes them: a masked gradient
              // keeps the sign of the rest of the product (+-0)
              const float up_mask = (U >= p.clamp_min && U <= p.clamp_max) ? 1.0f : 0.0f;
              const float gate_mask = (G <= p.clamp_max) ? 1.0f : 0.0f;
              x[i] = ref * pr * t * up_mask;                                                        // d up
              gv[i] = ref * pr * uo * sg * (1.0f + p.geglu_a * gc * (1.0f - sg)) * gate_mask;      // d gate
            }
          }
          output_chunk<IC, OUTC, !kPackedBwd>(p, x, row, xo, norm, lane, kblk_col, amax_local, os);
          output_chunk<IC, OUTC, !kPackedBwd>(p, gv, row, go, norm, lane, kblk_col, amax_local2, os);
          if (XC && p.dbias != nullptr && in_range(p.status, kSiteDbias, max(xo, go) + 31, p.n_out)) {
            float* db = p.dbias + static_cast<int64_t>(g) * p.n_out;
            add_column_sums32(x, db + xo, lane);
            add_column_sums32(gv, db + go, lane);
          }
        }
        if (kChunkLd) release();
        atomicAdd(p.dprob + row, dprob_local);
      } else if (EPI == EPI_SWIGLU) {
        const bool gf = p.gate_first != 0;
#pragma unroll
        for (int j = 0; j < kWarpCols / 64; ++j) {
          const int col0 = nt * (BN / 2) + e * (kWarpCols / 2) + 32 * j;
          if (col0 >= p.n_out) continue;
          if (kPairOnLoad) {
            epilogue_chunk<IC, EPI, OUTC, XC>(p, &r[64 * j], &r[64 * j + 32], row, col0, al_epi, pr, norm, lane,
                                               kblk_col, amax_local, seg_start, seg_rows, os);
          } else {
            uint32_t xs[32], gs[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              xs[i] = gf ? r[64 * j + 32 + i] : r[64 * j + i];
              gs[i] = gf ? r[64 * j + i] : r[64 * j + 32 + i];
            }
            epilogue_chunk<IC, EPI, OUTC, XC>(p, xs, gs, row, col0, al_epi, pr, norm, lane, kblk_col, amax_local,
                                               seg_start, seg_rows, os);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < kWarpCols / 32; ++c) {
          const int col0 = nt * BN + e * kWarpCols + 32 * c;
          if (col0 >= p.n_out) continue;
          epilogue_chunk<IC, EPI, OUTC, XC>(p, &r[32 * c], &r[32 * c], row, col0, al_epi, pr, norm, lane,
                                             kblk_col, amax_local, seg_start, seg_rows, os);
        }
      }
      if (OUTC == OUTC_FLOAT && p.amax != nullptr) {
        // backward: amax[2g] over the input-gradient blocks, amax[2g + 1] over
        // the gate-gradient blocks
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, o));
        const int ai = is_bwd_inst(EPI) ? 2 * g : g;
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.amax) + ai, __float_as_uint(amax_local));
        if (is_bwd_inst(EPI)) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            amax_local2 = fmaxf(amax_local2, __shfl_xor_sync(0xffffffffu, amax_local2, o));
          if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.amax) + ai + 1, __float_as_uint(amax_local2));
        }
      }
    }
    // every TMA store of this warp has completed (its staging slot is shared
    // memory that ends with the CTA)
    if (os.slot != 0u && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  if (CLUSTER) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, Ly::kTmemCols);
    else tmem_dealloc(tmem_base, Ly::kTmemCols);
  }
}

}  // namespace bsgg
