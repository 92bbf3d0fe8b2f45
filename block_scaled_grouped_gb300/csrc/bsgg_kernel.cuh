// bsgg_kernel.cuh -- the persistent grouped block-scaled GEMM kernel for sm_103a.
//
// One CTA per SM walks a static list of 128 x BN output tiles.  Tiles never
// straddle two expert groups because groups are padded to multiples of 128 rows
// ("Grouped GEMM + Quant (SM100)", Tiling and Cluster: tiles must not span
// groups).  Six warps per CTA:
//   warp 0      TMA producer: A, B[g] tiles (128-byte swizzle) and the 512-byte
//               scale-factor atoms (bulk copies) into a multi-stage ring
//   warp 1      tensor-memory allocator and MMA issuer: copies the stage's scale
//               atoms to tensor memory (tcgen05.cp) and issues block-scaled
//               tcgen05.mma (MXFP8 kind::mxf8f6f4 or NVFP4 kind::mxf4nvf4) into
//               one of NUM_ACC fp32 accumulators in tensor memory
//   warps 2..9  epilogue, two warps per 32-lane tensor-memory quadrant, each
//               taking every other 32-column chunk: tcgen05.ld, alpha, the
//               activation and prob (Step 2), then per-group amax or the row /
//               column block quantization (Step 3), and global stores
// All waits are bounded; a wait that runs out raises a CTA-wide abort flag and
// a device status bit, and every role then drains its in-flight asynchronous
// work (again with a bound) and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace bsgg {

enum : int { EPI_GATE = 0, EPI_SWIGLU = 1, EPI_SRELU = 2 };
// Output class (template) and exact output kind (runtime) of D.
enum : int { OUTC_FLOAT = 0, OUTC_FP8 = 1, OUTC_FP4 = 2 };
enum : int { OK_BF16 = 0, OK_F16 = 1, OK_F32 = 2, OK_E4M3 = 3, OK_E5M2 = 4, OK_E2M1 = 5 };

constexpr int kBM = 128;          // rows per tile (TMEM lanes)
constexpr int kBKBytes = 128;     // K bytes per pipeline stage (one 128-byte swizzle span)
constexpr int kEpiWarps = 8;     // two warps per tensor-memory lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxGroups = 1024;
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadOffsets = 2u;
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s per wait
constexpr uint64_t kDrainLimitNs = 200000000ull;     // 0.2 s per drain wait

struct Params {
  const uint8_t* sfa;
  const uint8_t* sfb;
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
  int32_t num_n_tiles, num_k_stages, num_tiles;
  int32_t raster_w;         // n-tiles per raster band inside a group
  int32_t kq_in;            // 512-byte SF atoms per 128 rows along K
  int32_t rn_b;             // 128-row SF row-blocks of one expert's B: ceil(N/128)
  int32_t kq_row;           // SF atoms per 128 rows of SFD_row: ceil(ceil(n_out/v)/4)
  int32_t kq_col;           // SF atoms per 128 columns of SFD_col: ceil(ceil(m_pad/v)/4)
  int32_t out_kind;         // OK_*
  int32_t want_col;
  int32_t gate_first;
  float tanh_s, tanh_rcp_s; // soft clamp s and 1/s (s = 0: off)
  float rcp_qmax;           // fp32(1/q_max) of the output format
  uint32_t idesc;           // tcgen05 instruction descriptor without scale ids
};

template <bool FP4, int BN>
struct Layout {
  static constexpr int kHalves = BN / 128;                 // 128-row SF blocks of a B tile
  static constexpr int kAtoms = FP4 ? 4 : 1;               // SF atoms per stage per 128 rows
  static constexpr int kKElems = FP4 ? 256 : 128;          // K elements per stage
  static constexpr int kMmaK = FP4 ? 64 : 32;              // K elements per MMA instruction
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = BN * kBKBytes;
  static constexpr int kSfaBytes = kAtoms * 512;
  static constexpr int kSfbBytes = kAtoms * kHalves * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStages = (221184 / kStageBytes) > 8 ? 8 : (221184 / kStageBytes);
  static constexpr int kNumAcc = (BN == 128) ? 2 : 1;
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
  static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1;
  static constexpr int kOffTmemHolder = kOffBars + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemHolder + 4;
  static constexpr int kOffOffsets = kOffAbort + 12;
  static constexpr int kSmemBytes = kOffOffsets + 4 * kMaxGroups + 1024;   // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffSfa % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

// Byte offset of the scale of (row, k-block) in a swizzled SF buffer whose
// rows hold kq 512-byte atoms: 128-row block, then k-atom, then inside the atom
// 16 bytes per row-in-32, 4 bytes per 32-row quarter, 1 byte per k-block.
__device__ __forceinline__ int64_t sf_off(int64_t row, int64_t kblk, int64_t kq) {
  return ((row >> 7) * kq + (kblk >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kblk & 3);
}

// Tile t of the static schedule -> (group, m-tile, n-tile).  Tiles of group g
// occupy [num_n_tiles * ms_g, num_n_tiles * me_g) where [ms_g, me_g) are the
// group's 128-row tiles; inside a group the n-tiles are walked in bands of
// raster_w, all m-tiles of a band before the next band, so that a band of B
// stays in L2 while every m-tile of the group passes over it.  Empty groups
// own no tiles.
__device__ __forceinline__ bool decode_tile(int t, const Params& p, const int32_t* s_off, int& g,
                                            int& m_tile, int& n_tile) {
  const int ntn = p.num_n_tiles;
  const int row = (t / ntn) * kBM;
  int lo = 0, hi = p.L;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] > row) hi = mid; else lo = mid + 1;
  }
  if (lo >= p.L) return false;
  g = lo;
  const int ms = (g ? s_off[g - 1] : 0) / kBM;
  const int mtg = s_off[g] / kBM - ms;
  const int r = t - ms * ntn;
  const int W = p.raster_w;
  const int band = r / (mtg * W);
  const int w = min(W, ntn - band * W);
  const int rr = r - band * mtg * W;
  m_tile = ms + rr / w;
  n_tile = band * W + rr % w;
  return true;
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

// 32 values of one row -> quantized codes stored at `dst` (32 bytes for FP8,
// 16 bytes for FP4), each value multiplied by its block's scale first.
template <int OUTC>
__device__ __forceinline__ void store_q32(void* dst, const float (&v)[32], const float (&sc)[32],
                                          int out_kind) {
  if (OUTC == OUTC_FP8) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t lo, hi;
      if (out_kind == OK_E4M3) {
        lo = cvt_e4m3x2(v[4 * i] * sc[4 * i], v[4 * i + 1] * sc[4 * i + 1]);
        hi = cvt_e4m3x2(v[4 * i + 2] * sc[4 * i + 2], v[4 * i + 3] * sc[4 * i + 3]);
      } else {
        lo = cvt_e5m2x2(v[4 * i] * sc[4 * i], v[4 * i + 1] * sc[4 * i + 1]);
        hi = cvt_e5m2x2(v[4 * i + 2] * sc[4 * i + 2], v[4 * i + 3] * sc[4 * i + 3]);
      }
      w[i] = lo | (hi << 16);
    }
    st_v4(dst, w[0], w[1], w[2], w[3]);
    st_v4(static_cast<uint8_t*>(dst) + 16, w[4], w[5], w[6], w[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 8 * i + 2 * j;
        x |= cvt_e2m1x2(v[e] * sc[e], v[e + 1] * sc[e + 1]) << (8 * j);
      }
      w[i] = x;
    }
    st_v4(dst, w[0], w[1], w[2], w[3]);
  }
}

template <bool FP4, int BN, int EPI, int OUTC>
__global__ void __launch_bounds__(kThreads, 1)
    bsgg_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ Params p) {
  using Ly = Layout<FP4, BN>;
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
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Ly::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kOffAbort);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + Ly::kOffOffsets);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < p.L; i += kThreads) s_off[i] = p.offsets[i];
  if (tid == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int a = 0; a < NA; ++a) { mbar_init(accf_bar(a), 1); mbar_init(acce_bar(a), kEpiWarps); }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Ly::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // padded_offsets must be non-decreasing multiples of 128 ending at m_pad.
  int bad = 0;
  for (int i = tid; i < p.L; i += kThreads) {
    const int prev = i ? s_off[i - 1] : 0;
    if (s_off[i] < prev || (s_off[i] % kBM) != 0) bad = 1;
  }
  if (tid == 0 && s_off[p.L - 1] != p.m_pad) bad = 1;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.status, kStatusBadOffsets);
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[S];
      bool issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) { issued[s] = false; issued_phase[s] = 0; }
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int g, mt, nt;
        if (!decode_tile(t, p, s_off, g, mt, nt)) continue;
        const uint8_t* sfa_tile = p.sfa + static_cast<int64_t>(mt) * p.kq_in * 512;
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs)) { ok = false; break; }
          const int atoms = min(Ly::kAtoms, p.kq_in - ks * Ly::kAtoms);
          int halves = 0;
#pragma unroll
          for (int h = 0; h < Ly::kHalves; ++h) halves += (nt * BN + 128 * h < p.n) ? 1 : 0;
          const uint32_t bytes = Ly::kABytes + Ly::kBBytes + atoms * 512u * (1 + halves);
          const uint32_t fb = full_bar(stage);
          mbar_expect_tx(fb, bytes);
          tma_load_2d(sbase + Ly::kOffA + stage * Ly::kABytes, &tmA, fb, ks * kBKBytes, mt * kBM);
          tma_load_3d(sbase + Ly::kOffB + stage * Ly::kBBytes, &tmB, fb, ks * kBKBytes, nt * BN, g);
          bulk_load(sbase + Ly::kOffSfa + stage * Ly::kSfaBytes, sfa_tile + ks * Ly::kAtoms * 512,
                    atoms * 512u, fb);
          for (int h = 0; h < halves; ++h) {
            const int64_t rb = static_cast<int64_t>(g) * p.rn_b + nt * Ly::kHalves + h;
            bulk_load(sbase + Ly::kOffSfb + stage * Ly::kSfbBytes + h * Ly::kAtoms * 512,
                      p.sfb + (rb * p.kq_in + ks * Ly::kAtoms) * 512, atoms * 512u, fb);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        // drain: wait (bounded) for every load this thread issued to land
        for (int s = 0; s < S; ++s)
          if (issued[s]) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(full_bar(s), issued_phase[s]) && globaltimer_ns() - t0 < kDrainLimitNs) {}
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t sf_tmem0 = tmem_base + NA * BN;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int g, mt, nt;
        if (!decode_tile(t, p, s_off, g, mt, nt)) continue;
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        int halves = 0;
#pragma unroll
        for (int h = 0; h < Ly::kHalves; ++h) halves += (nt * BN + 128 * h < p.n) ? 1 : 0;
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, kWaitLimitNs)) { ok = false; break; }
          tc_fence_after();
          const int atoms = min(Ly::kAtoms, p.kq_in - ks * Ly::kAtoms);
          const uint32_t sfa_t = sf_tmem0 + stage * Ly::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + Ly::kSfaCols;
          const uint32_t sfa_s = sbase + Ly::kOffSfa + stage * Ly::kSfaBytes;
          const uint32_t sfb_s = sbase + Ly::kOffSfb + stage * Ly::kSfbBytes;
          // scale atoms -> tensor memory: atom i of A at columns 4i; atom i of
          // B half h at columns 4*(i*halves_max + h)
          for (int i = 0; i < atoms; ++i) {
            tc_cp_32x128b_x4(sfa_t + 4 * i, sdesc_sf_block(sfa_s + 512 * i));
            for (int h = 0; h < halves; ++h)
              tc_cp_32x128b_x4(sfb_t + 4 * (i * Ly::kHalves + h),
                               sdesc_sf_block(sfb_s + (h * Ly::kAtoms + i) * 512));
          }
          const int k_left = p.k - ks * Ly::kKElems;
          const int n_mma = min(4, (k_left + Ly::kMmaK - 1) / Ly::kMmaK);
          const uint32_t a_s = sbase + Ly::kOffA + stage * Ly::kABytes;
          const uint32_t b_s = sbase + Ly::kOffB + stage * Ly::kBBytes;
          for (int kk = 0; kk < n_mma; ++kk) {
            const uint64_t ad = sdesc_kmajor_sw128(a_s + 32 * kk);
            const uint64_t bd = sdesc_kmajor_sw128(b_s + 32 * kk);
            const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
            if (FP4) {
              // one MMA consumes four 16-element blocks: a whole atom per row
              tc_mma_nvf4(d_tmem, ad, bd, p.idesc, sfa_t + 4 * kk, sfb_t + 4 * Ly::kHalves * kk, accum);
            } else {
              // one MMA consumes one 32-element block: byte kk of each row's word
              const uint32_t id = p.idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
              tc_mma_mxf8(d_tmem, ad, bd, id, sfa_t, sfb_t, accum);
            }
          }
          tc_commit(empty_bar(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));
        if (++acc == NA) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        // drain: wait (bounded) until every issued tcgen05 operation completed
        tc_commit(drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < kDrainLimitNs) {}
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // tensor-memory lane quadrant
    const int e = (warp - 2) >> 2;                // which of the quadrant's two warps
    const float norm = (OUTC == OUTC_FLOAT) ? 1.0f : *p.norm_const;
    int acc = 0;
    uint32_t acc_phase = 0;
    constexpr int kChunks = (EPI == EPI_SWIGLU) ? BN / 64 : BN / 32;
    constexpr int kOutPerTile = (EPI == EPI_SWIGLU) ? BN / 2 : BN;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int g, mt, nt;
      if (!decode_tile(t, p, s_off, g, mt, nt)) continue;
      const bool got = __all_sync(0xffffffffu, mbar_wait(accf_bar(acc), acc_phase, abort_flag, kWaitLimitNs));
      if (!got) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int row = mt * kBM + q * 32 + lane;
      const float pr = p.prob[row];
      const float al = p.alpha[g];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      float amax_local = 0.0f;
      for (int ch = e; ch < kChunks; ch += 2) {
        uint32_t ra[32], rb[32];
        if (EPI == EPI_SWIGLU) {
          const int cx = ch * 64 + (p.gate_first ? 32 : 0);
          const int cg = ch * 64 + (p.gate_first ? 0 : 32);
          tmem_ld32(taddr + cx, ra);
          tmem_ld32(taddr + cg, rb);
        } else {
          tmem_ld32(taddr + ch * 32, ra);
        }
        tmem_wait_ld();
        if (ch + 2 >= kChunks) {
          // this warp's part of the accumulator is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(acc));
        }
        const int col0 = nt * kOutPerTile + ch * 32;  // first D column of this chunk
        if (col0 >= p.n_out) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float c = al * __uint_as_float(ra[i]);
          if (EPI == EPI_GATE) {
            v[i] = pr * c;
          } else if (EPI == EPI_SRELU) {
            float r = fmaxf(c, 0.0f);
            if (p.tanh_s > 0.0f) r = p.tanh_s * fminf(tanh_approx(r * p.tanh_rcp_s), 1.0f);
            v[i] = pr * (r * r);
          } else {
            const float gt = al * __uint_as_float(rb[i]);
            const float sig = __fdividef(1.0f, 1.0f + __expf(-gt));
            v[i] = pr * c * (gt * sig);
          }
        }
        if (OUTC == OUTC_FLOAT) {
#pragma unroll
          for (int i = 0; i < 32; ++i) amax_local = fmaxf(amax_local, fabsf(v[i]));
          if (p.out_kind == OK_F32) {
            float* dst = static_cast<float*>(p.d) + static_cast<int64_t>(row) * p.n_out + col0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_v4(dst + 4 * i, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                    __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
          } else {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (p.out_kind == OK_BF16) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
              } else {
                __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
              }
            }
            uint16_t* dst = static_cast<uint16_t*>(p.d) + static_cast<int64_t>(row) * p.n_out + col0;
#pragma unroll
            for (int i = 0; i < 4; ++i) st_v4(dst + 8 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        } else {
          // ---- row blocks (v = 32 for UE8M0 scales, 16 for E4M3 scales)
          constexpr int kV = FP4 ? 16 : 32;
          const int64_t row_bytes = (OUTC == OUTC_FP8) ? p.n_out : p.n_out / 2;
          const int64_t col_byte0 = (OUTC == OUTC_FP8) ? col0 : col0 / 2;
          float sc[32];
#pragma unroll
          for (int b = 0; b < 32 / kV; ++b) {
            float am = 0.0f;
#pragma unroll
            for (int i = 0; i < kV; ++i) am = fmaxf(am, fabsf(v[b * kV + i]));
            uint32_t code;
            float s;
            block_scale<FP4>(am, norm, p.rcp_qmax, code, s);
#pragma unroll
            for (int i = 0; i < kV; ++i) sc[b * kV + i] = s;
            p.sfd_row[sf_off(row, col0 / kV + b, p.kq_row)] = static_cast<uint8_t>(code);
          }
          store_q32<OUTC>(static_cast<uint8_t*>(p.d) + row * row_bytes + col_byte0, v, sc, p.out_kind);
          // ---- column blocks: 32 rows = the 32 lanes of this warp (v = 32)
          if (!FP4 && p.want_col) {
            // column j's max over the warp's 32 rows; lane j keeps it, encodes
            // that column's scale and shares the factor with the other lanes
            float my_am = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float am = __uint_as_float(redux_max_u32(__float_as_uint(fabsf(v[j]))));
              my_am = (lane == j) ? am : my_am;
            }
            uint32_t my_code;
            float my_scale;
            block_scale<false>(my_am, norm, p.rcp_qmax, my_code, my_scale);
#pragma unroll
            for (int j = 0; j < 32; ++j) sc[j] = __shfl_sync(0xffffffffu, my_scale, j);
            store_q32<OUTC>(static_cast<uint8_t*>(p.d_col) + row * row_bytes + col_byte0, v, sc, p.out_kind);
            p.sfd_col[sf_off(col0 + lane, mt * 4 + q, p.kq_col)] = static_cast<uint8_t>(my_code);
          }
        }
      }
      if (OUTC == OUTC_FLOAT && p.amax != nullptr) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, o));
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.amax) + g, __float_as_uint(amax_local));
      }
      if (++acc == NA) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Ly::kTmemCols);
  }
}

}  // namespace bsgg
