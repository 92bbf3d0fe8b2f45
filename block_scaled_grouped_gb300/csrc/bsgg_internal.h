// bsgg_internal.h -- declarations shared by the host ABI and the kernel
// instantiation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "bsgg_kernel.cuh"

namespace bsgg {

struct Launch {
  CUtensorMap tmA;
  CUtensorMap tmB;
  Params p;
  int grid;
  int bn;
  int epi;
  int outc;
  cudaStream_t stream;
};

// Launchers, one per input family (separate translation units so that the
// instantiations compile in parallel).  Return the launch's cudaError_t.
cudaError_t launch_mxf8(const Launch& L);
cudaError_t launch_nvf4(const Launch& L);
// Dynamic shared memory a launch of this family needs.
int smem_bytes(bool fp4, int bn);

}  // namespace bsgg
