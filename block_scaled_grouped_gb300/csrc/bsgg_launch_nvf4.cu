// Kernel instances for NVFP4 inputs (E2M1 data, E4M3 scales per 16).
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_nvf4(const Launch& L) { return launch_family<true>(L); }
int smem_bytes(bool fp4, int bn) {
  if (bn != 128) return 0;
  return fp4 ? Layout<true, 128>::kSmemBytes : Layout<false, 128>::kSmemBytes;
}
}  // namespace bsgg
