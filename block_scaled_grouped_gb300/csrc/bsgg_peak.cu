// bsgg_peak.cu -- bsgg_measure_mma_peak: the dense block-scaled tensor-core
// throughput of this GPU, the denominator of the kernel's roofline.
//
// One CTA per SM keeps A (128 x 128 bytes), B (BN x 128 bytes) and unit
// scale factors resident in shared memory and issues nothing but
// tcgen05.mma ... block_scale (MXFP8: kind::mxf8f6f4, K = 32; NVFP4:
// kind::mxf4nvf4, K = 64), four per 128-byte K slice, into one tensor-memory
// accumulator.  No loads, no epilogue: what remains is the tensor pipe.
#include <cstdint>

#include "../../include/bsgg.h"
#include "ptx.cuh"

namespace {

using namespace bsgg;

constexpr int kPeakThreads = 128;
constexpr uint64_t kPeakWaitNs = 2000000000ull;

template <bool FP4, int BN>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int64_t iters, uint32_t idesc, uint32_t* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done_bar;
  __shared__ uint32_t holder;
  constexpr int kOpBytes = 16384 + BN * 128;        // A then B, 128-byte swizzled rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // finite operand codes from a hash (E4M3: exponent field <= 14; any E2M1
  // nibble is finite), unit scales (UE8M0 127 = 1.0, E4M3 0x38 = 1.0)
  for (int i = threadIdx.x; i < kOpBytes; i += kPeakThreads) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u + blockIdx.x * 97u;
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    sm[i] = static_cast<uint8_t>(h & 0x77u);
  }
  for (int i = threadIdx.x; i < 6144; i += kPeakThreads) sm[kOpBytes + i] = FP4 ? 0x38 : 127;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&holder), 512);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> MMA reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = holder;
  if (warp == 0 && lane == 0) {
    const uint32_t a_s = smem_u32(sm), b_s = a_s + 16384, sf_s = a_s + kOpBytes;
    const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 256 + 16;
    // scale atoms: 4 for A (one per NVFP4 MMA; MXFP8 uses the first), 2 x 4 for B
    for (int i = 0; i < 4; ++i) tc_cp_32x128b_x4(sfa_t + 4 * i, sdesc_sf_block(sf_s + 512 * i));
    for (int i = 0; i < 8; ++i) tc_cp_32x128b_x4(sfb_t + 4 * i, sdesc_sf_block(sf_s + 2048 + 512 * (i & 3)));
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
        if (FP4) tc_mma_nvf4(tmem, ad[kk], bd[kk], id[kk], sfa_t + 4 * kk, sfb_t + 4 * (BN / 128) * kk, 1u);
        else tc_mma_mxf8(tmem, ad[kk], bd[kk], id[kk], sfa_t, sfb_t, 1u);
      }
    }
    tc_commit(smem_u32(&done_bar));
    const uint64_t t0 = globaltimer_ns();
    bool ok = false;
    while (!(ok = mbar_try_wait(smem_u32(&done_bar), 0)) && globaltimer_ns() - t0 < kPeakWaitNs) {}
    if (!ok) atomicOr(status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

uint32_t peak_idesc(bool fp4, int bn) {
  const uint32_t fmt = fp4 ? 1u : 0u, ue8m0 = fp4 ? 0u : 1u;
  return (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(bn >> 3) << 17) | (ue8m0 << 23) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

template <bool FP4, int BN>
cudaError_t launch_peak(int sms, int64_t iters, uint32_t* status, cudaStream_t s) {
  auto k = mma_peak_kernel<FP4, BN>;
  const int smem = 1024 + 16384 + BN * 128 + 6144;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<sms, kPeakThreads, smem, s>>>(iters, peak_idesc(FP4, BN), status);
  return cudaGetLastError();
}

}  // namespace

extern "C" bsgg_status bsgg_measure_mma_peak(int32_t in_format, int32_t tile_n, int64_t mmas_per_sm,
                                             double* tflops, void* stream) {
  // at most 2^22 MMAs per SM: well under a second, inside the kernel's 2 s wait
  if (!tflops || (tile_n != 128 && tile_n != 256) || mmas_per_sm < 4 || mmas_per_sm > (int64_t(1) << 22))
    return BSGG_ERR_INVALID_ARG;
  if (in_format < BSGG_IN_MXFP8_E4M3 || in_format > BSGG_IN_NVFP4) return BSGG_ERR_INVALID_ARG;
  const bool fp4 = in_format == BSGG_IN_NVFP4;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BSGG_ERR_CUDA;
  uint32_t* status = nullptr;
  if (cudaMalloc(&status, sizeof(uint32_t)) != cudaSuccess) return BSGG_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bsgg_status st = BSGG_OK;
  const int64_t iters = mmas_per_sm / 4;
  auto launch = [&](int64_t n) -> cudaError_t {
    if (fp4) return tile_n == 256 ? launch_peak<true, 256>(sms, n, status, s) : launch_peak<true, 128>(sms, n, status, s);
    return tile_n == 256 ? launch_peak<false, 256>(sms, n, status, s) : launch_peak<false, 128>(sms, n, status, s);
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
    const double flops = 2.0 * 128.0 * tile_n * (fp4 ? 64.0 : 32.0) * 4.0 * double(iters) * sms;
    *tflops = flops / (double(ms) * 1e-3) / 1e12;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(status);
  return st;
}
