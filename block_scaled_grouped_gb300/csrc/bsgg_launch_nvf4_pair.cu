// Kernel instances of the forward epilogues: NVFP4 inputs (E2M1 data, E4M3 scales per 16), 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_nvf4_pair(const Launch& L) { return launch_shape_fwd<IC_NVF4, 256, CM_PAIR>(L); }
int cluster_resident_ctas(bool fp4) {
  return fp4 ? cluster_resident_ctas_impl<IC_NVF4>() : cluster_resident_ctas_impl<IC_MXF8>();
}
}  // namespace bsgg
