// bsgg_launch.cuh -- instantiates the kernel for one (input family, tile
// shape, cluster mode) and dispatches a Launch to the right (epilogue, output
// class) instance.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include "bsgg_internal.h"

namespace bsgg {

template <int IC, int BN, int CM, int EPI, int OUTC, bool XC>
cudaError_t launch_one(const Launch& L) {
  auto kern = bsgg_kernel<IC, BN, CM, EPI, OUTC, XC>;
  constexpr bool FP4 = ic_fp4(IC);
  constexpr bool kCluster = CM != CM_SINGLE;
  constexpr bool kStores = scale_stores<FP4>();
  using Ro = Roles<kStores>;
  const int smem = Layout<FP4, BN, CM == CM_PAIR, ic_scaled(IC), stage_slices(IC, CM)>::kSmemBytes;
  // The function attributes are set once per device and instance.  Bit d of
  // `configured` says device d is done; host threads that launch this instance
  // at the same time serialise on the mutex until the bit is set.
  static std::atomic<uint64_t> configured{0};
  static std::mutex configure_mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t(1) << dev;
  if ((configured.load(std::memory_order_acquire) & bit) == 0) {
    std::lock_guard<std::mutex> lk(configure_mu);
    if ((configured.load(std::memory_order_relaxed) & bit) == 0) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      if (kCluster) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
      }
      if (kStores) {
        // the warpgroups' setmaxnreg shares add up to exactly the launch's
        // registers only if the kernel was compiled to kLaunchRegs per thread;
        // with fewer the raising warps would wait forever: refuse to launch
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != Ro::kLaunchRegs) return cudaErrorInvalidConfiguration;
      }
      configured.fetch_or(bit, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(L.grid), 1, 1);
  cfg.blockDim = dim3(Ro::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  if (kCluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmSFA, L.tmSFB, L.tmD, L.tmDcol, L.p);
}

template <int IC, int BN, int CM, int EPI, bool XC>
cudaError_t launch_outc(const Launch& L) {
  // bfloat16 operands (the BF16 backend): 16/32-bit outputs only
  if constexpr (IC == IC_BF16) {
    return L.outc == OUTC_FLOAT ? launch_one<IC, BN, CM, EPI, OUTC_FLOAT, XC>(L) : cudaErrorInvalidValue;
  } else {
    switch (L.outc) {
      case OUTC_FLOAT: return launch_one<IC, BN, CM, EPI, OUTC_FLOAT, XC>(L);
      case OUTC_FP8:
        // FP8 outputs come from MXFP8 inputs only (the host refuses them for FP4)
        if constexpr (ic_fp4(IC)) return cudaErrorInvalidValue;
        else return launch_one<IC, BN, CM, EPI, OUTC_FP8, XC>(L);
      case OUTC_FP4: return launch_one<IC, BN, CM, EPI, OUTC_FP4, XC>(L);
    }
    return cudaErrorInvalidValue;
  }
}

// The XC instances: forward launches with a bias, a stored C or the Hadamard
// output; backward launches with dbias.
template <int IC, int BN, int CM, int EPI>
cudaError_t launch_xc(const Launch& L) {
  const bool xc = is_bwd_inst(EPI) ? L.p.dbias != nullptr
                                   : (L.p.bias != nullptr || L.p.c_out != nullptr || L.p.rht != nullptr);
  return xc ? launch_outc<IC, BN, CM, EPI, true>(L) : launch_outc<IC, BN, CM, EPI, false>(L);
}

// Forward epilogues (one translation unit per input family and tile shape) and
// backward epilogues (another), so that the instances compile in parallel.
template <int IC, int BN, int CM>
cudaError_t launch_shape_fwd(const Launch& L) {
  switch (L.epi) {
    case EPI_GATE: return launch_xc<IC, BN, CM, EPI_GATE>(L);
    case EPI_SWIGLU: return launch_xc<IC, BN, CM, EPI_SWIGLU>(L);
    case EPI_SRELU: return launch_xc<IC, BN, CM, EPI_SRELU>(L);
  }
  return cudaErrorInvalidValue;
}
template <int IC, int BN, int CM>
cudaError_t launch_shape_bwd(const Launch& L) {
  switch (L.epi) {
    case EPI_DSWIGLU: return launch_xc<IC, BN, CM, EPI_DSWIGLU>(L);
    case EPI_DSITUGLU:
      // dSiTU-GLU is not a BF16-backend activation
      if constexpr (IC == IC_BF16) return cudaErrorInvalidValue;
      else return launch_xc<IC, BN, CM, EPI_DSITUGLU>(L);
  }
  return cudaErrorInvalidValue;
}

// CTA pairs of this kernel that fit on the device at once, x 2.
template <int IC>
int cluster_resident_ctas_impl() {
  constexpr bool FP4 = ic_fp4(IC);
  auto kern = bsgg_kernel<IC, 256, CM_PAIR, EPI_GATE, OUTC_FLOAT, false>;
  const int smem = Layout<FP4, 256, true, true, stage_slices(IC, CM_PAIR)>::kSmemBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(Roles<scale_stores<FP4>()>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) return 0;
  return 2 * clusters;
}

}  // namespace bsgg
