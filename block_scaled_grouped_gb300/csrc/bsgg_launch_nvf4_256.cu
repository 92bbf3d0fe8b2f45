// Kernel instances of the forward epilogues: NVFP4 inputs (E2M1 data, E4M3 scales per 16), 1-CTA 128 x 256 tiles.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_nvf4_256(const Launch& L) { return launch_shape_fwd<IC_NVF4, 256, CM_SINGLE>(L); }
}  // namespace bsgg
