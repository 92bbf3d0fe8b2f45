// bsgg_peak.cu -- bsgg_measure_mma_peak(_tile): the dense block-scaled
// tensor-core throughput of this GPU, the denominator of the kernel's roofline.
//
// Every SM keeps A (128 x 128 bytes), its share of B and unit scale factors
// resident in shared memory and issues nothing but tcgen05.mma ... block_scale
// (MXFP8: kind::mxf8f6f4, K = 32; NVFP4: kind::mxf4nvf4, K = 64), four per
// 128-byte K slice, into one tensor-memory accumulator.  No loads, no
// epilogue: what remains is the tensor pipe.  Two instruction forms, the two
// the GEMM kernel issues:
//   * cta_group::1, M = 128, N = 128 or 256: one CTA per SM issues its own MMAs;
//   * cta_group::2, M = 256, N = 256: a cluster of two CTAs (an SM pair), each
//     holding its 128 rows of A and half of B's 256 rows; the even CTA issues
//     every MMA of the pair.
#include <cstdint>

#include "../../include/bsgg.h"
#include "ptx.cuh"

namespace {

using namespace bsgg;

constexpr int kPeakThreads = 128;
constexpr uint64_t kPeakWaitNs = 2000000000ull;
constexpr int kPeakSfBytes = 6144;                   // 4 A atoms + 8 B atoms of 512 bytes

template <int BN, bool PAIR>
constexpr int peak_op_bytes() { return 16384 + (PAIR ? BN / 2 : BN) * 128; }   // A then this CTA's B rows

template <bool FP4, int BN, bool PAIR>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int64_t iters, uint32_t idesc, uint32_t* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done_bar;
  __shared__ uint32_t holder;
  constexpr int kOpBytes = peak_op_bytes<BN, PAIR>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool issues = !PAIR || cluster_ctarank() == 0;
  // finite operand codes from a hash (E4M3: exponent field <= 14; any E2M1
  // nibble is finite), unit scales (UE8M0 127 = 1.0, E4M3 0x38 = 1.0)
  for (int i = threadIdx.x; i < kOpBytes; i += kPeakThreads) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u + blockIdx.x * 97u;
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    sm[i] = static_cast<uint8_t>(h & 0x77u);
  }
  for (int i = threadIdx.x; i < kPeakSfBytes; i += kPeakThreads) sm[kOpBytes + i] = FP4 ? 0x38 : 127;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    if (PAIR) { tmem_alloc_pair(smem_u32(&holder), 512); tmem_relinquish_pair(); }
    else { tmem_alloc(smem_u32(&holder), 512); tmem_relinquish(); }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> MMA reads
  tc_fence_before();
  // a pair's MMAs read both CTAs' shared memory and commit to both CTAs'
  // barriers: both must be initialised first
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = holder;
  if (warp == 0 && lane == 0) {
    bool ok = true;
    if (issues) {
      const uint32_t a_s = smem_u32(sm), b_s = a_s + 16384, sf_s = a_s + kOpBytes;
      const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 256 + 16;
      // scale atoms: 4 for A (one per NVFP4 MMA; MXFP8 uses the first), 2 x 4
      // for B; a pair's copies fill each CTA's tensor memory from its own
      // shared memory
      for (int i = 0; i < 4; ++i) {
        if (PAIR) tc_cp_32x128b_x4_pair(sfa_t + 4 * i, sdesc_sf_block(sf_s + 512 * i));
        else tc_cp_32x128b_x4(sfa_t + 4 * i, sdesc_sf_block(sf_s + 512 * i));
      }
      for (int i = 0; i < 8; ++i) {
        if (PAIR) tc_cp_32x128b_x4_pair(sfb_t + 4 * i, sdesc_sf_block(sf_s + 2048 + 512 * (i & 3)));
        else tc_cp_32x128b_x4(sfb_t + 4 * i, sdesc_sf_block(sf_s + 2048 + 512 * (i & 3)));
      }
      uint64_t ad[4], bd[4];
      uint32_t id[4];
      for (int kk = 0; kk < 4; ++kk) {
        ad[kk] = sdesc_kmajor_sw128(a_s + 32 * kk);
        bd[kk] = sdesc_kmajor_sw128(b_s + 32 * kk);
        id[kk] = FP4 ? idesc : (idesc | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4));
      }
      for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t sb = sfb_t + 4 * (BN / 128) * kk;
          if (FP4) {
            if (PAIR) tc_mma_nvf4_pair(tmem, ad[kk], bd[kk], id[kk], sfa_t + 4 * kk, sb, 1u);
            else tc_mma_nvf4(tmem, ad[kk], bd[kk], id[kk], sfa_t + 4 * kk, sb, 1u);
          } else {
            if (PAIR) tc_mma_mxf8_pair(tmem, ad[kk], bd[kk], id[kk], sfa_t, sfb_t, 1u);
            else tc_mma_mxf8(tmem, ad[kk], bd[kk], id[kk], sfa_t, sfb_t, 1u);
          }
        }
      }
      // completion arrives on the barrier of every CTA of the pair
      if (PAIR) tc_commit_pair(smem_u32(&done_bar), 3); else tc_commit(smem_u32(&done_bar));
    }
    const uint64_t t0 = globaltimer_ns();
    while (!(ok = mbar_try_wait(smem_u32(&done_bar), 0)) && globaltimer_ns() - t0 < kPeakWaitNs) {}
    if (!ok) atomicOr(status, 1u);
  }
  tc_fence_before();
  if (PAIR) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, 512); else tmem_dealloc(tmem, 512);
  }
}

uint32_t peak_idesc(bool fp4, int bn, bool pair) {
  const uint32_t fmt = fp4 ? 1u : 0u, ue8m0 = fp4 ? 0u : 1u;
  return (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(bn >> 3) << 17) | (ue8m0 << 23) |
         (static_cast<uint32_t>((pair ? 256 : 128) >> 4) << 24);
}

template <bool FP4, int BN, bool PAIR>
cudaError_t launch_peak(int sms, int64_t iters, uint32_t* status, cudaStream_t s) {
  auto k = mma_peak_kernel<FP4, BN, PAIR>;
  // more than half of an SM's shared memory: one CTA per SM, so that no CTA
  // waits on another's tensor-memory allocation
  constexpr int kNeed = 1024 + peak_op_bytes<BN, PAIR>() + kPeakSfBytes;
  const int smem = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? (sms / 2) * 2 : sms), 1, 1);
  cfg.blockDim = dim3(kPeakThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, k, iters, peak_idesc(FP4, BN, PAIR), status);
}

}  // namespace

extern "C" bsgg_status bsgg_measure_mma_peak_tile(int32_t in_format, int32_t tile_m, int32_t tile_n,
                                                  int64_t mmas, double* tflops, void* stream) {
  // at most 2^22 MMAs per issuing thread: well under a second, inside the
  // kernel's 2 s wait
  if (!tflops || (tile_n != 128 && tile_n != 256) || mmas < 4 || mmas > (int64_t(1) << 22))
    return BSGG_ERR_INVALID_ARG;
  if (tile_m != 128 && tile_m != 256) return BSGG_ERR_INVALID_ARG;
  if (tile_m == 256 && tile_n != 256) return BSGG_ERR_UNSUPPORTED;   // pairs: 256 x 256, as in the GEMM
  if (in_format < BSGG_IN_MXFP8_E4M3 || in_format > BSGG_IN_NVFP4) return BSGG_ERR_INVALID_ARG;
  const bool fp4 = in_format == BSGG_IN_NVFP4;
  const bool pair = tile_m == 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BSGG_ERR_CUDA;
  if (pair && sms < 2) return BSGG_ERR_UNSUPPORTED;
  uint32_t* status = nullptr;
  if (cudaMalloc(&status, sizeof(uint32_t)) != cudaSuccess) return BSGG_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bsgg_status st = BSGG_OK;
  const int64_t iters = mmas / 4;
  auto launch = [&](int64_t n) -> cudaError_t {
    if (pair) return fp4 ? launch_peak<true, 256, true>(sms, n, status, s) : launch_peak<false, 256, true>(sms, n, status, s);
    if (fp4) return tile_n == 256 ? launch_peak<true, 256, false>(sms, n, status, s)
                                  : launch_peak<true, 128, false>(sms, n, status, s);
    return tile_n == 256 ? launch_peak<false, 256, false>(sms, n, status, s)
                         : launch_peak<false, 128, false>(sms, n, status, s);
  };
  float ms = 0.0f;
  uint32_t word = 0;
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess || launch(iters / 10 + 1) != cudaSuccess ||
      cudaEventRecord(e0, s) != cudaSuccess || launch(iters) != cudaSuccess || cudaEventRecord(e1, s) != cudaSuccess ||
      cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
      cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    st = BSGG_ERR_CUDA;
  } else if (word != 0) {
    st = BSGG_ERR_DEVICE_TIMEOUT;
  } else {
    // 2 M N K per instruction; one issuing thread per SM, or per SM pair
    const double issuers = pair ? double(sms / 2) : double(sms);
    const double flops = 2.0 * tile_m * tile_n * (fp4 ? 64.0 : 32.0) * 4.0 * double(iters) * issuers;
    *tflops = flops / (double(ms) * 1e-3) / 1e12;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(status);
  return st;
}

extern "C" bsgg_status bsgg_measure_mma_peak(int32_t in_format, int32_t tile_n, int64_t mmas_per_sm,
                                             double* tflops, void* stream) {
  return bsgg_measure_mma_peak_tile(in_format, 128, tile_n, mmas_per_sm, tflops, stream);
}
