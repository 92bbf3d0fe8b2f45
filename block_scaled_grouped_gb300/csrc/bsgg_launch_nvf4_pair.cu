// Kernel instances: NVFP4 inputs (E2M1 data, E4M3 scales per 16), 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_nvf4_pair(const Launch& L) { return launch_shape<true, 256, true>(L); }
int pair_resident_ctas(bool fp4) {
  return fp4 ? pair_resident_ctas_impl<true>() : pair_resident_ctas_impl<false>();
}
}  // namespace bsgg
