// Kernel instances of the backward epilogues: NVFP4 inputs (E2M1 data, E4M3 scales per 16), 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_nvf4_pair_bwd(const Launch& L) { return launch_shape_bwd<IC_NVF4, 256, CM_PAIR>(L); }
}  // namespace bsgg
