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
  CUtensorMap tmSFA;
  CUtensorMap tmSFB;
  CUtensorMap tmD;      // D and D_col as (row bytes, m_pad) byte tensors, boxes of one 32-row chunk
  CUtensorMap tmDcol;   // (zero where the output is not stored through TMA)
  Params p;
  int grid;      // CTAs (a multiple of 2 for clusters)
  int bn;        // 128 or 256
  bool pair;     // 256 x 256 tiles on a CTA pair
  int epi;
  int outc;
  cudaStream_t stream;
};

// Launchers, one translation unit per (input family, tile shape) so that the
// instantiations compile in parallel.  Return the launch's cudaError_t.
cudaError_t launch_mxf8_128(const Launch& L);
cudaError_t launch_mxf8_256(const Launch& L);
cudaError_t launch_mxf8_pair(const Launch& L);
cudaError_t launch_nvf4_128(const Launch& L);
cudaError_t launch_nvf4_256(const Launch& L);
cudaError_t launch_nvf4_pair(const Launch& L);
cudaError_t launch_f4e8_128(const Launch& L);
cudaError_t launch_f4e8_256(const Launch& L);
cudaError_t launch_f4e8_pair(const Launch& L);
// the same for the backward epilogues
cudaError_t launch_mxf8_128_bwd(const Launch& L);
cudaError_t launch_mxf8_256_bwd(const Launch& L);
cudaError_t launch_mxf8_pair_bwd(const Launch& L);
cudaError_t launch_nvf4_128_bwd(const Launch& L);
cudaError_t launch_nvf4_256_bwd(const Launch& L);
cudaError_t launch_nvf4_pair_bwd(const Launch& L);
cudaError_t launch_f4e8_128_bwd(const Launch& L);
cudaError_t launch_f4e8_256_bwd(const Launch& L);
cudaError_t launch_f4e8_pair_bwd(const Launch& L);
cudaError_t launch_bf16_128_bwd(const Launch& L);
cudaError_t launch_bf16_256_bwd(const Launch& L);
cudaError_t launch_bf16_pair_bwd(const Launch& L);
// Largest number of CTAs of the CTA-pair kernel that can be resident at once
// (clusters x 2) on the current device, 0 if unknown.
int cluster_resident_ctas(bool fp4);

}  // namespace bsgg
