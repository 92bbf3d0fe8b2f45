// bsgg_launch.cuh -- instantiates the kernel for one input family and
// dispatches a Launch to the right (BN, epilogue, output class) instance.
#pragma once

#include "bsgg_internal.h"

namespace bsgg {

template <bool FP4, int BN, int EPI, int OUTC>
cudaError_t launch_one(const Launch& L) {
  auto kern = bsgg_kernel<FP4, BN, EPI, OUTC>;
  const int smem = Layout<FP4, BN>::kSmemBytes;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kern<<<L.grid, kThreads, smem, L.stream>>>(L.tmA, L.tmB, L.p);
  return cudaGetLastError();
}

template <bool FP4, int BN, int EPI>
cudaError_t launch_outc(const Launch& L) {
  switch (L.outc) {
    case OUTC_FLOAT: return launch_one<FP4, BN, EPI, OUTC_FLOAT>(L);
    case OUTC_FP8: return launch_one<FP4, BN, EPI, OUTC_FP8>(L);
    case OUTC_FP4: return launch_one<FP4, BN, EPI, OUTC_FP4>(L);
  }
  return cudaErrorInvalidValue;
}

template <bool FP4, int BN>
cudaError_t launch_epi(const Launch& L) {
  switch (L.epi) {
    case EPI_GATE: return launch_outc<FP4, BN, EPI_GATE>(L);
    case EPI_SWIGLU: return launch_outc<FP4, BN, EPI_SWIGLU>(L);
    case EPI_SRELU: return launch_outc<FP4, BN, EPI_SRELU>(L);
  }
  return cudaErrorInvalidValue;
}

template <bool FP4>
cudaError_t launch_family(const Launch& L) {
  if (L.bn == 128) return launch_epi<FP4, 128>(L);
  return cudaErrorInvalidValue;
}

}  // namespace bsgg
